// Blackwell tensor-core helpers (sm_103a): TMA tensor loads, shared-memory
// matrix descriptors, tcgen05 MMA with the accumulator in tensor memory.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace lora {

// ------------------------------------------------------------ TMA tensor --

// 2-D tiled TMA load of the box at (c0 = innermost, c1) into shared memory,
// completing as transaction bytes on `bar`.  c0 * element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// The same load multicast to the CTAs of the cluster in `mask`: the box lands at
// offset `dst` of each one's shared memory and completes on its barrier at `bar`.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar,
                                               uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "h"(mask)
      : "memory");
}

// 2-D tiled TMA store of the shared-memory box at `src` to (c0 = innermost, c1),
// tracked in this thread's bulk-async group.  The box must lie inside the
// tensor; c0 * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int c0, int c1, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's bulk stores have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until this thread's bulk stores are complete (their writes performed).
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (the tensor cores and TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte global -> shared copy (LSU async copy); `valid == false` writes zeros
// without reading the source.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid = true) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// Close this thread's current group of cp.async copies (wait_group counts groups).
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// ----------------------------------------------------- matrix descriptors --

// Shared-memory matrix descriptor for tcgen05.mma:
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride-dimension byte offset >> 4
//   bits 46-47 descriptor version (1 on this architecture)
//   bits 49-51 base offset (0: every swizzle atom starts 1024-byte aligned)
//   bits 61-63 layout: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16: fp32 accumulator, bf16 A and
// B, A K-major, B K-major (b_mn_major = 0) or MN-major (1), shape M x N.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15 A major, 16 B major, 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// -------------------------------------------------------------- tcgen05 --

// Allocate `ncols` tensor-memory columns (a power of two >= 32); one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every MMA issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Arrive once on the barrier at `bar` in each CTA of the cluster in `mask` when
// every MMA issued so far by this thread completes.
__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 16 columns of 32-bit accumulator: thread i of the warp receives
// lane (taddr.lane + i), columns taddr.col .. +15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 32 columns, without waiting: call tmem_wait_ld() before using r.
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival counts toward the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a tile laid
// out in the 128-byte-swizzle canonical form (rows of 128 bytes, 8-row atoms of
// 1024 bytes, chunk index XOR row % 8) -- the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B into a 1024-byte-aligned buffer.
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// bf16 matrix [rows, cols] with a row stride of `ld` elements as a tensor map
// of box_rows x 64 boxes with 128-byte swizzle (host).  False when the driver
// offers no encoder or rejects the map; the kernels then copy every tile row by
// row.
bool make_act_map(CUtensorMap* m, const void* base, long long rows, long long cols, long long ld, int box_rows);

// ------------------------------------------------------- long tiles --

constexpr int kTM = LORA_TILE_M;  // 128

// One long tile: rows p0 .. p0 + cnt - 1 of the segment order, all on adapter ad.
struct TileInfo {
  int ad, p0, cnt;
  int row0;  // token of the first row
  bool tma;  // 128 consecutive tokens and tensor maps available
};

__device__ __forceinline__ TileInfo load_tile(const int32_t* long_units, const int32_t* seg_adapter,
                                              const int32_t* indptr, const int32_t* perm, int tile, int use_tma) {
  TileInfo t;
  const int s = long_units[2 * tile], m0 = long_units[2 * tile + 1];
  t.ad = seg_adapter[s];
  t.p0 = indptr[s] + m0;
  t.cnt = min(kTM, indptr[s + 1] - t.p0);
  t.row0 = perm[t.p0];
  t.tma = use_tma && t.cnt == kTM && perm[t.p0 + kTM - 1] - t.row0 == kTM - 1;
  return t;
}

// Adapter id, rank, every page-list slot and page of A_i and B_i, checked by
// one warp; returns 0 or LORA_DERR_* bits (the same in every lane).  `d` is
// adapter_desc(v, ad).
__device__ __forceinline__ int check_adapter_warp(const DevView& v, int ad, const lora_adapter_desc_t& d, int lane) {
  if (ad < 0 || ad >= v.n_adapters) return LORA_DERR_BAD_ADAPTER;
  if (d.rank < 1 || d.rank > v.max_rank || d.rank > LORA_MAX_RANK) return LORA_DERR_BAD_RANK;
  const long long na = ((long long)d.rank * v.d_in + (1LL << v.page_shift) - 1) >> v.page_shift;
  const long long nb = ((long long)d.rank * v.d_out + (1LL << v.page_shift) - 1) >> v.page_shift;
  int mine = 0;
  for (long long i0 = 0; i0 < na + nb; i0 += 32 * 8) {  // eight page-list reads in flight per lane
    int pv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const long long i = i0 + 32 * k + lane;
      const long long slot = i < na ? d.a_page0 + i : d.b_page0 + (i - na);
      pv[k] = 0;
      if (i < na + nb) pv[k] = (slot < 0 || slot >= v.n_page_list) ? -1 : v.page_list[slot];
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (pv[k] < 0 || pv[k] >= v.n_pages) mine = 1;
  }
  return __any_sync(0xffffffffu, mine) ? LORA_DERR_BAD_PAGE : 0;
}

}  // namespace lora
