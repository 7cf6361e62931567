// sm103a_ptx.cuh -- thin inline-PTX wrappers for the Blackwell features the kernels use:
// mbarriers, TMA tensor loads, tensor memory (tcgen05.alloc/ld/st) and tcgen05.mma.
// Written from the public PTX ISA; each wrapper is one instruction or a bounded loop around one.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fattn {

// ---------------------------------------------------------------------------------------------
// Debug builds (compiled with -DFATTN_DEBUG).  The wrappers below check their operands against
// rules the hardware enforces before they issue: shared-memory and barrier alignment, TMA
// coordinates (the innermost coordinate of a tiled copy must address a multiple of 16 bytes, and a
// store or reduce may not start at a negative coordinate), the 32-lane quarter of tensor memory a
// warp may access and the 512 columns each kernel allocates.  A broken rule is recorded in the
// translation unit's debug record (the rule's bit, and the first failure's block, thread and rule)
// and the instruction is not issued, so a bad operand is reported instead of faulting the GPU; a
// copy left out leaves its barrier incomplete, and the bounded waits then end the kernel.  Kernels
// check their global stores against their outputs' extents the same way.  The host reads the
// records with fattn_debug_take.  Release builds compile every check out.
// ---------------------------------------------------------------------------------------------
enum DebugRule : uint32_t {
  kDbgSmemAlign = 1u << 0,  // shared-memory operand or barrier address not aligned
  kDbgTmaCoord = 1u << 1,   // TMA innermost coordinate not a multiple of 16 elements, or a store/reduce below 0
  kDbgTmemLane = 1u << 2,   // tcgen05.ld/st/mma address outside the lanes the warp (or the MMA) may use
  kDbgTmemCol = 1u << 3,    // tensor-memory columns past the 512 allocated
  kDbgBulk = 1u << 4,       // untiled bulk copy: size or global address not a multiple of 16 bytes
  kDbgGlobal = 1u << 5,     // a kernel's global store outside its output
};
constexpr uint32_t kTmemColumns = 512;

// The rules as pure functions of the operands (host and device): each returns the rules the
// operands break, 0 when they break none.  Every TMA coordinate this library issues along the
// innermost dimension is a multiple of 16 elements, which is 16-byte aligned for every element
// size it uses (1, 2 and 4 bytes); tiled copies land on 128-byte aligned shared memory.
__host__ __device__ constexpr uint32_t dbg_bar(uint32_t bar) { return (bar & 7u) ? kDbgSmemAlign : 0u; }
__host__ __device__ constexpr uint32_t dbg_tma_tile(uint32_t smem, uint32_t bar, int x, int y, int z, bool store) {
  return ((smem & 127u) ? kDbgSmemAlign : 0u) | (store ? 0u : dbg_bar(bar)) | ((x & 15) ? kDbgTmaCoord : 0u) |
         ((store && (x < 0 || y < 0 || z < 0)) ? kDbgTmaCoord : 0u);
}
__host__ __device__ constexpr uint32_t dbg_bulk(uint32_t smem, uint64_t gaddr, uint32_t bytes, uint32_t bar) {
  return ((smem & 15u) ? kDbgSmemAlign : 0u) | dbg_bar(bar) |
         (((gaddr & 15u) || (bytes & 15u) || bytes == 0u) ? kDbgBulk : 0u);
}
// tcgen05.ld/st by warp `warp` of its CTA: lanes 32 (warp % 4) .. + 31, columns [col, col + cols).
__host__ __device__ constexpr uint32_t dbg_tmem(uint32_t taddr, uint32_t cols, uint32_t warp) {
  return ((taddr >> 16) != 32u * (warp & 3u) ? kDbgTmemLane : 0u) |
         ((taddr & 0xFFFFu) + cols > kTmemColumns ? kDbgTmemCol : 0u);
}
// tcgen05.mma with M = 128: the accumulator starts at lane 0 and spans the instruction's N columns
// (N / 8 in bits 17-22 of the instruction descriptor).
__host__ __device__ constexpr uint32_t dbg_mma_d(uint32_t d_tmem, uint32_t idesc) {
  return ((d_tmem >> 16) != 0u ? kDbgTmemLane : 0u) |
         ((d_tmem & 0xFFFFu) + ((idesc >> 17) & 0x3Fu) * 8u > kTmemColumns ? kDbgTmemCol : 0u);
}
static_assert(dbg_tma_tile(1024, 8, 64, -3, 0, false) == 0 && dbg_tma_tile(1040, 8, 0, 0, 0, false) == kDbgSmemAlign &&
                  dbg_tma_tile(1024, 12, 0, 0, 0, false) == kDbgSmemAlign &&
                  dbg_tma_tile(1024, 8, 8, 0, 0, false) == kDbgTmaCoord &&
                  dbg_tma_tile(1024, 0, 32, -1, 0, true) == kDbgTmaCoord && dbg_tma_tile(1024, 0, 32, 5, 2, true) == 0,
              "TMA rules");
static_assert(dbg_bulk(16, 32, 4096, 8) == 0 && dbg_bulk(8, 32, 4096, 8) == kDbgSmemAlign &&
                  dbg_bulk(16, 40, 4096, 8) == kDbgBulk && dbg_bulk(16, 32, 4100, 8) == kDbgBulk,
              "bulk rules");
static_assert(dbg_tmem((64u << 16) | 480u, 32, 6) == 0 && dbg_tmem((64u << 16) | 481u, 32, 6) == kDbgTmemCol &&
                  dbg_tmem((32u << 16), 32, 6) == kDbgTmemLane && dbg_tmem((96u << 16) | 16u, 16, 11) == 0,
              "tensor-memory rules");
static_assert(dbg_mma_d(384u, (128u >> 3) << 17) == 0 && dbg_mma_d(448u, (128u >> 3) << 17) == kDbgTmemCol &&
                  dbg_mma_d((32u << 16) | 0u, (64u >> 3) << 17) == kDbgTmemLane,
              "MMA accumulator rules");

#ifdef FATTN_DEBUG
// This translation unit's debug record.
static __device__ unsigned int g_fattn_dbg_rules;        // OR of the rules broken
static __device__ unsigned long long g_fattn_dbg_first;  // first failure: block << 32 | thread << 8 | rule + 1
static __device__ __noinline__ void dbg_record(uint32_t rules) {
  atomicOr(&g_fattn_dbg_rules, rules);
  const unsigned long long rec = (static_cast<unsigned long long>(blockIdx.x) << 32) |
                                 (static_cast<unsigned long long>(threadIdx.x) << 8) |
                                 static_cast<unsigned long long>(__ffs(static_cast<int>(rules)));
  atomicCAS(&g_fattn_dbg_first, 0ull, rec);
}
static __device__ __forceinline__ bool dbg_fails(uint32_t rules) {
  if (rules == 0u) return false;
  dbg_record(rules);
  return true;
}
// Skip the rest of the calling wrapper when its operands break a rule.
#define FATTN_DBG_SKIP_IF(rules) \
  if (::fattn::dbg_fails(rules)) return
// A global store of element `index` into an output of `count` elements: false (recorded) outside.
static __device__ __forceinline__ bool dbg_in(long long index, long long count) {
  return !dbg_fails(index >= 0 && index < count ? 0u : kDbgGlobal);
}
// Host accessor of the record, defined once in each translation unit that has kernels.
#define FATTN_DEBUG_ACCESSOR(name)                                                                      \
  cudaError_t debug_take_##name(unsigned int* rules, unsigned long long* first, bool clear) {           \
    cudaError_t e = cudaMemcpyFromSymbol(rules, g_fattn_dbg_rules, sizeof(unsigned int));             \
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(first, g_fattn_dbg_first, sizeof(unsigned long long)); \
    if (e == cudaSuccess && clear) {                                                                  \
      const unsigned int r0 = 0u;                                                                     \
      const unsigned long long f0 = 0ull;                                                             \
      e = cudaMemcpyToSymbol(g_fattn_dbg_rules, &r0, sizeof r0);                                      \
      if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fattn_dbg_first, &f0, sizeof f0);                \
    }                                                                                                 \
    return e;                                                                                         \
  }
#else
#define FATTN_DBG_SKIP_IF(rules)
static __device__ __forceinline__ constexpr bool dbg_in(long long, long long) { return true; }
#define FATTN_DEBUG_ACCESSOR(name)                                                            \
  cudaError_t debug_take_##name(unsigned int* rules, unsigned long long* first, bool) {       \
    *rules = 0u;                                                                            \
    *first = 0ull;                                                                          \
    return cudaSuccess;                                                                     \
  }
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  FATTN_DBG_SKIP_IF(dbg_bar(bar));
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  FATTN_DBG_SKIP_IF(dbg_bar(bar));
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  FATTN_DBG_SKIP_IF(dbg_bar(bar));
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
#ifdef FATTN_DEBUG
  if (dbg_fails(dbg_bar(bar))) return true;  // reported, not waited on
#endif
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, but never forever: the loop gives up when
// the CTA's abort word is set by another thread, or when `deadline_ns` of the global timer has
// passed.  Returns true on completion, false on giving up (the caller then winds down).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile uint32_t* abort_flag,
                                                  uint64_t deadline_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (((++spins) & 63u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() > deadline_ns) return false;
    }
  }
}

// ---------------------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), 3-D tiled loads completing on an mbarrier
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                            int y, int z) {
  FATTN_DBG_SKIP_IF(dbg_tma_tile(dst, bar, x, y, z, false));
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Untiled bulk copy global -> shared completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  FATTN_DBG_SKIP_IF(dbg_bulk(dst, reinterpret_cast<uint64_t>(src), bytes, bar));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Element-wise fp32 add of a shared-memory box into global memory through a 3-D tensor map
// (TMA reduce); tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  FATTN_DBG_SKIP_IF(dbg_tma_tile(src, 0u, x, y, z, true));
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk group of this thread has finished reading its shared source.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make this thread's generic-proxy shared-memory writes visible to the async proxy (tcgen05.mma
// operand reads, TMA stores and reduces).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `nthreads` threads that also returns the OR of every thread's predicate.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------------------------
// Tensor memory
// ---------------------------------------------------------------------------------------------
// Whole warp: allocate `ncols` TMEM columns (power of two >= 32); the base address is written to
// shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Warp-wide: each lane reads 32 consecutive 32-bit columns of its own TMEM lane.  The lane field
// of `taddr` must be the warp's 32-lane quarter.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
#ifdef FATTN_DEBUG
  if (dbg_fails(dbg_tmem(taddr, 32, threadIdx.x >> 5))) {
    for (int i = 0; i < 32; ++i) r[i] = 0u;
    return;
  }
#endif
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Warp-wide: each lane reads 64 consecutive 32-bit columns of its own TMEM lane in one instruction.
__device__ __forceinline__ void tmem_ld_32x32b_x64(uint32_t taddr, uint32_t (&r)[2][32]) {
#ifdef FATTN_DEBUG
  if (dbg_fails(dbg_tmem(taddr, 64, threadIdx.x >> 5))) {
    for (int h = 0; h < 2; ++h)
      for (int i = 0; i < 32; ++i) r[h][i] = 0u;
    return;
  }
#endif
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(r[0][0]), "=r"(r[0][1]), "=r"(r[0][2]), "=r"(r[0][3]), "=r"(r[0][4]), "=r"(r[0][5]), "=r"(r[0][6]), "=r"(r[0][7]),
        "=r"(r[0][8]), "=r"(r[0][9]), "=r"(r[0][10]), "=r"(r[0][11]), "=r"(r[0][12]), "=r"(r[0][13]), "=r"(r[0][14]), "=r"(r[0][15]),
        "=r"(r[0][16]), "=r"(r[0][17]), "=r"(r[0][18]), "=r"(r[0][19]), "=r"(r[0][20]), "=r"(r[0][21]), "=r"(r[0][22]), "=r"(r[0][23]),
        "=r"(r[0][24]), "=r"(r[0][25]), "=r"(r[0][26]), "=r"(r[0][27]), "=r"(r[0][28]), "=r"(r[0][29]), "=r"(r[0][30]), "=r"(r[0][31]),
        "=r"(r[1][0]), "=r"(r[1][1]), "=r"(r[1][2]), "=r"(r[1][3]), "=r"(r[1][4]), "=r"(r[1][5]), "=r"(r[1][6]), "=r"(r[1][7]),
        "=r"(r[1][8]), "=r"(r[1][9]), "=r"(r[1][10]), "=r"(r[1][11]), "=r"(r[1][12]), "=r"(r[1][13]), "=r"(r[1][14]), "=r"(r[1][15]),
        "=r"(r[1][16]), "=r"(r[1][17]), "=r"(r[1][18]), "=r"(r[1][19]), "=r"(r[1][20]), "=r"(r[1][21]), "=r"(r[1][22]), "=r"(r[1][23]),
        "=r"(r[1][24]), "=r"(r[1][25]), "=r"(r[1][26]), "=r"(r[1][27]), "=r"(r[1][28]), "=r"(r[1][29]), "=r"(r[1][30]), "=r"(r[1][31])
      : "r"(taddr));
}

// Warp-wide: each lane reads 128 consecutive 32-bit columns of its own TMEM lane in one instruction
// (the four 32-column groups of a 128-key score row).
__device__ __forceinline__ void tmem_ld_32x32b_x128(uint32_t taddr, uint32_t (&r)[4][32]) {
#ifdef FATTN_DEBUG
  if (dbg_fails(dbg_tmem(taddr, 128, threadIdx.x >> 5))) {
    for (int h = 0; h < 4; ++h)
      for (int i = 0; i < 32; ++i) r[h][i] = 0u;
    return;
  }
#endif
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];"
      : "=r"(r[0][0]), "=r"(r[0][1]), "=r"(r[0][2]), "=r"(r[0][3]), "=r"(r[0][4]), "=r"(r[0][5]), "=r"(r[0][6]), "=r"(r[0][7]),
        "=r"(r[0][8]), "=r"(r[0][9]), "=r"(r[0][10]), "=r"(r[0][11]), "=r"(r[0][12]), "=r"(r[0][13]), "=r"(r[0][14]), "=r"(r[0][15]),
        "=r"(r[0][16]), "=r"(r[0][17]), "=r"(r[0][18]), "=r"(r[0][19]), "=r"(r[0][20]), "=r"(r[0][21]), "=r"(r[0][22]), "=r"(r[0][23]),
        "=r"(r[0][24]), "=r"(r[0][25]), "=r"(r[0][26]), "=r"(r[0][27]), "=r"(r[0][28]), "=r"(r[0][29]), "=r"(r[0][30]), "=r"(r[0][31]),
        "=r"(r[1][0]), "=r"(r[1][1]), "=r"(r[1][2]), "=r"(r[1][3]), "=r"(r[1][4]), "=r"(r[1][5]), "=r"(r[1][6]), "=r"(r[1][7]),
        "=r"(r[1][8]), "=r"(r[1][9]), "=r"(r[1][10]), "=r"(r[1][11]), "=r"(r[1][12]), "=r"(r[1][13]), "=r"(r[1][14]), "=r"(r[1][15]),
        "=r"(r[1][16]), "=r"(r[1][17]), "=r"(r[1][18]), "=r"(r[1][19]), "=r"(r[1][20]), "=r"(r[1][21]), "=r"(r[1][22]), "=r"(r[1][23]),
        "=r"(r[1][24]), "=r"(r[1][25]), "=r"(r[1][26]), "=r"(r[1][27]), "=r"(r[1][28]), "=r"(r[1][29]), "=r"(r[1][30]), "=r"(r[1][31]),
        "=r"(r[2][0]), "=r"(r[2][1]), "=r"(r[2][2]), "=r"(r[2][3]), "=r"(r[2][4]), "=r"(r[2][5]), "=r"(r[2][6]), "=r"(r[2][7]),
        "=r"(r[2][8]), "=r"(r[2][9]), "=r"(r[2][10]), "=r"(r[2][11]), "=r"(r[2][12]), "=r"(r[2][13]), "=r"(r[2][14]), "=r"(r[2][15]),
        "=r"(r[2][16]), "=r"(r[2][17]), "=r"(r[2][18]), "=r"(r[2][19]), "=r"(r[2][20]), "=r"(r[2][21]), "=r"(r[2][22]), "=r"(r[2][23]),
        "=r"(r[2][24]), "=r"(r[2][25]), "=r"(r[2][26]), "=r"(r[2][27]), "=r"(r[2][28]), "=r"(r[2][29]), "=r"(r[2][30]), "=r"(r[2][31]),
        "=r"(r[3][0]), "=r"(r[3][1]), "=r"(r[3][2]), "=r"(r[3][3]), "=r"(r[3][4]), "=r"(r[3][5]), "=r"(r[3][6]), "=r"(r[3][7]),
        "=r"(r[3][8]), "=r"(r[3][9]), "=r"(r[3][10]), "=r"(r[3][11]), "=r"(r[3][12]), "=r"(r[3][13]), "=r"(r[3][14]), "=r"(r[3][15]),
        "=r"(r[3][16]), "=r"(r[3][17]), "=r"(r[3][18]), "=r"(r[3][19]), "=r"(r[3][20]), "=r"(r[3][21]), "=r"(r[3][22]), "=r"(r[3][23]),
        "=r"(r[3][24]), "=r"(r[3][25]), "=r"(r[3][26]), "=r"(r[3][27]), "=r"(r[3][28]), "=r"(r[3][29]), "=r"(r[3][30]), "=r"(r[3][31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  FATTN_DBG_SKIP_IF(dbg_tmem(taddr, 32, threadIdx.x >> 5));
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  FATTN_DBG_SKIP_IF(dbg_tmem(taddr, 16, threadIdx.x >> 5));
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// ---------------------------------------------------------------------------------------------
// tcgen05.mma, kind::f16 (bf16 x bf16 -> fp32), one CTA
// ---------------------------------------------------------------------------------------------
// Instruction descriptor: D fp32, A and B bf16, dense, M x N; `b_mn_major` selects an MN-major
// (N-contiguous) B operand and `a_mn_major` an MN-major (M-contiguous) A operand in shared memory.
__host__ __device__ constexpr uint32_t mma_idesc_bf16_f32(int M, int N, bool b_mn_major, bool a_mn_major = false) {
  return (1u << 4)                                   // D format: fp32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)            // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
         | ((static_cast<uint32_t>(N) >> 3) << 17)   // N / 8
         | ((static_cast<uint32_t>(M) >> 4) << 24);  // M / 16
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand whose 8-row x 128-byte swizzle
// atoms are laid out with the given leading/stride byte offsets.  `addr` is a shared-window byte
// address.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version for tcgen05
  d |= 2ull << 61;  // 128-byte swizzle
  return d;
}

// Descriptor for a K-major operand with 64-byte swizzle: rows of 64 bytes (64 e4m3, two K steps of
// kind::f8f6f4), 8-row atoms of 512 bytes stacked along M/N; the atom must start on a 512-byte boundary.
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;    // leading byte offset (unused: K fits in one swizzle span)
  d |= static_cast<uint64_t>(512u >> 4) << 32;
  d |= 1ull << 46;
  d |= 4ull << 61;  // 64-byte swizzle
  return d;
}

// Descriptor for a K-major operand with 32-byte swizzle: rows of 32 bytes (16 bf16, one K step),
// 8-row atoms of 256 bytes stacked along M/N.
__device__ __forceinline__ uint64_t smem_desc_sw32(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;    // leading byte offset (unused within one K step)
  d |= static_cast<uint64_t>(256u >> 4) << 32;
  d |= 1ull << 46;
  d |= 6ull << 61;  // 32-byte swizzle
  return d;
}

// D[tmem] (+)= A[smem] * B[smem]^T
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  FATTN_DBG_SKIP_IF(dbg_mma_d(d_tmem, idesc));
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  FATTN_DBG_SKIP_IF(dbg_mma_d(d_tmem, idesc) | ((a_tmem & 0xFFFFu) + 8u > kTmemColumns ? kDbgTmemCol : 0u));
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Warp-wide forms: every lane executes the instruction stream with the same (warp-uniform)
// operands and only the lane whose `lead` is non-zero issues.  Keeping the whole warp on one
// straight-line path lets the operands stay in uniform registers, so back-to-back MMAs issue at the
// tensor core's own rate.
__device__ __forceinline__ void mma_ss_lead(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate, uint32_t lead) {
  FATTN_DBG_SKIP_IF(dbg_mma_d(d_tmem, idesc));
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(lead)
      : "memory");
}

__device__ __forceinline__ void mma_ts_lead(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate, uint32_t lead) {
  FATTN_DBG_SKIP_IF(dbg_mma_d(d_tmem, idesc) | ((a_tmem & 0xFFFFu) + 8u > kTmemColumns ? kDbgTmemCol : 0u));
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(lead)
      : "memory");
}

__device__ __forceinline__ void mma_commit_lead(uint32_t bar, uint32_t lead) {
  FATTN_DBG_SKIP_IF(dbg_bar(bar));
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
      "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
      "r"(lead)
      : "memory");
}

// Lane-election for the warp-wide forms: non-zero in exactly one lane of a converged warp.
__device__ __forceinline__ uint32_t elect_lane() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred;
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  FATTN_DBG_SKIP_IF(dbg_bar(bar));
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// ---------------------------------------------------------------------------------------------
// Math helpers
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

}  // namespace fattn
