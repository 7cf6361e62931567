"""Failure detection without a GPU fault.

Every wait in the prefill (bf16 and FP8) and backward kernels is bounded.  A wait that gives up sets the library's device
status word, and the kernel then winds down: in-flight copies land, MMAs drain, TMEM is freed.
The host reads the word with fattn_last_error.  The test makes one wait run out: a test-only switch
(FATTN_TEST_DROP_KV_BLOCK) stops the producer from loading one key tile, so nothing ever completes
that tile's barrier (FATTN_TEST_DROP_BWD_KV does the same for the backward's key and value
tiles).  The test then checks that the call returns, that the timeout is reported
exactly once, and that the context is still usable.  It runs in a child process because the
switches are read once per process.
"""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import math, sys
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np
import torch
import exact_attention_31_gb300 as fa
from exact_attention_31_gb300.workloads import make_qkv
from parity_utils import compare, oracle_full

q, k, v, _ = make_qkv(1, 2, 512, 512, 64, seed=7, device="cuda")
o, lse = fa.fattn_fwd(q, k, v)          # key tile 1 is never loaded
torch.cuda.synchronize()                # the kernel ended by itself; no CUDA error
assert fa.fattn_last_error() == fa.FATTN_ERR_TIMEOUT
assert fa.fattn_last_error() == fa.FATTN_OK   # read-and-clear

# the context is still usable and correct
dq, dk, dv, _ = make_qkv(1, 2, 1, 300, 64, seed=8, device="cuda")
od, ld = fa.fattn_decode(dq, dk, dv)
torch.cuda.synchronize()
o_ref, l_ref = oracle_full(dq, dk, dv, False, 1 / math.sqrt(64))
compare(od, ld, o_ref, l_ref, what="decode after a reported timeout")
assert fa.fattn_last_error() == fa.FATTN_OK
print("FAILURE-DETECTION-OK")
"""


CHILD_BWD = r"""
import math, sys
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
import torch
import exact_attention_31_gb300 as fa
from exact_attention_31_gb300.workloads import make_dout, make_qkv
from parity_utils import compare, oracle_full

q, k, v, _ = make_qkv(1, 2, 512, 512, 64, seed=9, device="cuda")
do = make_dout(1, 2, 512, 64, seed=9, device="cuda")
o, lse = fa.fattn_fwd(q, k, v, causal=True)        # the forward is untouched by the switch
torch.cuda.synchronize()
assert fa.fattn_last_error() == fa.FATTN_OK
fa.fattn_bwd(q, k, v, o, lse, do, causal=True)     # no key/value tile is ever loaded
torch.cuda.synchronize()
assert fa.fattn_last_error() == fa.FATTN_ERR_TIMEOUT
assert fa.fattn_last_error() == fa.FATTN_OK

o2, l2 = fa.fattn_fwd(q, k, v, causal=True)
torch.cuda.synchronize()
o_ref, l_ref = oracle_full(q, k, v, True, 1 / math.sqrt(64))
compare(o2, l2, o_ref, l_ref, what="forward after a reported backward timeout")
assert fa.fattn_last_error() == fa.FATTN_OK
print("FAILURE-DETECTION-BWD-OK")
"""


@pytest.mark.gpu
def test_backward_bounded_wait_reports_timeout_and_context_survives():
    env = dict(os.environ, FATTN_WAIT_TIMEOUT_MS="200", FATTN_TEST_DROP_BWD_KV="1")
    env.pop("FATTN_TEST_DROP_KV_BLOCK", None)
    r = subprocess.run([sys.executable, "-c", CHILD_BWD, ROOT], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAILURE-DETECTION-BWD-OK" in r.stdout


@pytest.mark.gpu
def test_bounded_wait_reports_timeout_and_context_survives():
    env = dict(os.environ, FATTN_WAIT_TIMEOUT_MS="200", FATTN_TEST_DROP_KV_BLOCK="1")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAILURE-DETECTION-OK" in r.stdout


CHILD_FP8 = r"""
import math, sys
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
import torch
import exact_attention_31_gb300 as fa
from exact_attention_31_gb300.workloads import make_qkv, make_qkv_fp8
from parity_utils import compare, oracle_full

d = int(sys.argv[2])
(q8, k8, v8), (qs, ks, vs), _ = make_qkv_fp8(1, 2, 512, 512, d, seed=11, device="cuda")
fa.fattn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True)   # key tile 1 is never loaded
torch.cuda.synchronize()
assert fa.fattn_last_error() == fa.FATTN_ERR_TIMEOUT
assert fa.fattn_last_error() == fa.FATTN_OK

dq, dk, dv, _ = make_qkv(1, 2, 1, 300, 128, seed=12, device="cuda")
od, ld = fa.fattn_decode(dq, dk, dv)
torch.cuda.synchronize()
o_ref, l_ref = oracle_full(dq, dk, dv, False, 1 / math.sqrt(128))
compare(od, ld, o_ref, l_ref, what="decode after a reported FP8 timeout")
assert fa.fattn_last_error() == fa.FATTN_OK
print("FAILURE-DETECTION-FP8-OK")
"""


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_fp8_bounded_wait_reports_timeout_and_context_survives(d):
    env = dict(os.environ, FATTN_WAIT_TIMEOUT_MS="200", FATTN_TEST_DROP_KV_BLOCK="1")
    r = subprocess.run([sys.executable, "-c", CHILD_FP8, ROOT, str(d)], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAILURE-DETECTION-FP8-OK" in r.stdout
