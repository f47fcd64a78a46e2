// Device helpers shared by the library's kernels: mbarriers, bulk (TMA) copies,
// thread-block-cluster barriers and distributed shared memory, bf16 packing.
// Target: sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lora_sgmv.h"

namespace lora {

// Device-side copy of lora_pool_view_t (a kernel parameter).
struct DevView {
  const uint16_t* pool;
  const int32_t* page_list;
  const lora_adapter_desc_t* adapters;
  long long n_pages;
  long long n_page_list;
  int n_adapters;
  int page_shift;  // log2(page_elems)
  int max_rank;
  int d_in;
  int d_out;
  // 1: the kernels see every adapter transposed (B_i in the role of A_i and the
  // other way round, d_in and d_out exchanged), for the backward pass
  int swap_ab;
};

// Roughly one second at the GB300's clocks: the bound on every spin-wait.
constexpr long long kWaitCycles = 2000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Test for completion of the phase with the given parity.  A waiting thread
// is suspended in hardware (woken when the phase completes, or after at most
// about a millisecond) instead of spinning, so waiting warps leave the issue
// slots and the shared-memory pipe to the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// if about a second passed without completion.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) return false;
  }
  return true;
}

// Bounded wait with an explicit limit in clock cycles (false when it ran out).
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// The timeout probe of the kernels (lora_debug_wait_probe): thread 0 of the CTA
// waits, for at most `limit` cycles, on a barrier of its own that nothing
// arrives on, no transaction bytes are expected on and no copy or peer store
// targets; true if the wait completed (it never does), false when it ran out.
// The CTA's threads read the verdict after a __syncthreads.
__device__ __forceinline__ bool wait_probe(uint64_t* bar, long long limit) {
  mbar_init(smem_u32(bar), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  return mbar_wait_for(smem_u32(bar), 0, limit);
}

// --------------------------------------------------- bulk copy (non-tensor TMA) --

// global -> shared copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) that signals completion as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- clusters --

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t ncluster_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// All threads of all CTAs of the cluster: release our shared-memory writes,
// acquire the peers'.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive once on the mbarrier at `cluster_addr` (possibly in a peer CTA),
// releasing this thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Bounded wait, with cluster-scope acquire, for the phase with the given
// parity of a barrier in this CTA that peers arrive on.  False after about a
// second without completion.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  long long t0 = 0;
  for (bool first = true;; first = false) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(1000000u)
        : "memory");
    if (done) return true;
    if (first) t0 = clock64();
    else if (clock64() - t0 > kWaitCycles) return false;
  }
}

__device__ __forceinline__ void st_dsmem_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Asynchronous 16-byte store into the shared memory of a CTA of the cluster
// (possibly this one); its bytes complete as transaction bytes on the
// mbarrier at `cluster_bar`, which sits in the same CTA as the destination.
// Whoever waits on that barrier sees the data once the phase completes.
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, const float4& v, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   cluster_addr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(cluster_bar)
               : "memory");
}

// ------------------------------------------------- programmatic dependent launch --

// Wait until the grids this one depends on have completed and their memory is
// visible, then let the next grid in the stream start its prologue.  Every
// kernel of the library calls this before its first global-memory access, so
// a kernel launched early (programmatic stream serialization) never reads or
// writes anything its predecessor still touches.
__device__ __forceinline__ void pdl_wait_then_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The same, or, when `after_independent` is set, only the release: for a grid
// launched right after a library kernel that itself waited for everything
// before it (its CTAs release their dependents only after that wait) and that
// touches none of this grid's data.  Everything this grid reads was then
// complete before it started.  Such a grid calls pdl_exit before it ends.
__device__ __forceinline__ void pdl_enter(bool after_independent) {
  if (!after_independent) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// For a grid that entered with pdl_enter(true): wait for the predecessor before
// ending, so that this grid's completion still implies its predecessor's and the
// grids after it (which wait only for this one) see every earlier write.  The
// predecessor's CTAs are all resident by then (they released this grid), so
// the wait cannot hold up their progress.
__device__ __forceinline__ void pdl_exit(bool after_independent) {
  if (after_independent) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------- bf16 --

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Round two fp32 values to bf16 (nearest, ties to even); `a` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
  f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
  f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
  f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

// The descriptor of adapter `ad`; a zero one (rank 0) when `ad` is outside
// [0, n_adapters) of the view, so nothing outside the descriptor array is read.
__device__ __forceinline__ lora_adapter_desc_t adapter_desc(const DevView& v, int ad) {
  lora_adapter_desc_t d{};
  if (ad >= 0 && ad < v.n_adapters) d = v.adapters[ad];
  if (v.swap_ab) {
    const int32_t t = d.a_page0;
    d.a_page0 = d.b_page0;
    d.b_page0 = t;
  }
  return d;
}

__device__ __forceinline__ void report(int32_t* err, int bits) {
  if (err != nullptr && bits) atomicOr(err, bits);
}

}  // namespace lora
