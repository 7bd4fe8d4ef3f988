// Device-side building blocks for the verify-and-sample kernels (sm_103a).
//
// Thread-block clusters and distributed shared memory (DSMEM), mbarrier-tracked
// bulk copies (the non-tensor TMA path) with bounded waits, Philox4x32-10,
// order-preserving logit keys, the exponent-binned softmax weights, exact
// fixed-point comparisons, and deterministic block-level reductions and scans.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace sv {

constexpr int NT = 256;             // threads per CTA
constexpr int NWARP = NT / 32;

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Full cluster barrier with release/acquire semantics on shared::cluster memory.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}
// Loads from a peer CTA's shared memory. They are ordered after cluster barriers
// (which are compiler memory barriers); no clobber here, so independent peer
// loads can be issued back to back.
__device__ __forceinline__ uint32_t ld_peer_u32(const void* p, uint32_t rank) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(peer_addr(p, rank)));
  return v;
}
__device__ __forceinline__ uint64_t ld_peer_u64(const void* p, uint32_t rank) {
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(peer_addr(p, rank)));
  return v;
}
__device__ __forceinline__ float ld_peer_f32(const void* p, uint32_t rank) {
  return __uint_as_float(ld_peer_u32(p, rank));
}

// ---------------------------------------------------------- mbarrier + bulk
__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Orders this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for phase `parity` of `bar` for at most `limit_ns`; false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}
// One bulk copy global -> this CTA's shared memory, completion counted on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, unsigned long long* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------ Philox
// Philox4x32-10 (Salmon et al., SC'11): ten rounds of two 32x32->64 multiplies,
// word permutation and key XOR, with the Weyl key bump between rounds.
struct U4 {
  uint32_t x, y, z, w;
};
__device__ __forceinline__ U4 philox4x32_10(U4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = U4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
  }
  return c;
}
// Uniforms for (sequence b, position i): word 0 -> acceptance, word 1 -> sampling.
// Returned as the 24-bit integer grid index k (uniform = k * 2^-24).
__device__ __forceinline__ void philox_uniform_bits(uint64_t seed, uint64_t offset, uint32_t b,
                                                    uint32_t i, uint32_t* ku, uint32_t* kv) {
  U4 r = philox4x32_10(U4{i, b, (uint32_t)offset, (uint32_t)(offset >> 32)}, (uint32_t)seed,
                       (uint32_t)(seed >> 32));
  *ku = r.x >> 8;
  *kv = r.y >> 8;
}

// -------------------------------------------------------------------- keys
// Order-preserving 32-bit key of a float logit; -0.0 and +0.0 share a key, so
// key order equals float order (ties are then broken by token id).
__device__ __forceinline__ uint32_t okey(float z) {
  uint32_t u = __float_as_uint(z);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// ------------------------------------------------------------ arithmetic
__device__ __forceinline__ float ex2_approx(float y) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
  return r;
}
// max that returns NaN if either input is NaN
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
// 2^k as a float for integer k (0 below the normal range)
__device__ __forceinline__ float pow2i(int k) {
  return k < -126 ? 0.0f : (k > 127 ? __int_as_float(0x7f800000) : __int_as_float((k + 127) << 23));
}
// floor(x * 2^k) for finite x >= 0 (0 for x below the normal range), built from
// the float's bits with integer shifts; exact (truncation toward zero). The
// result must fit 64 bits (x * 2^k < 2^64).
__device__ __forceinline__ unsigned long long fix_pow2(float x, int k) {
  const uint32_t b = __float_as_uint(x);
  const int E = (int)((b >> 23) & 0xFFu);
  if (E == 0 || (b >> 31)) return 0ull;
  const unsigned long long M = (unsigned long long)((b & 0x7FFFFFu) | 0x800000u);
  const int sh = E - 150 + k;                     // x * 2^k = M * 2^sh
  if (sh >= 0) return M << sh;
  if (sh <= -24) return 0ull;
  return M >> (-sh);
}
// 16- and 32-bit loads from shared memory by shared-window address.
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// 128-bit product compare: a*b > c*d for 64-bit unsigned operands.
__device__ __forceinline__ bool mul_gt(uint64_t a, uint64_t b, uint64_t c, uint64_t d) {
  const uint64_t ah = __umul64hi(a, b), al = a * b;
  const uint64_t ch = __umul64hi(c, d), cl = c * d;
  return ah > ch || (ah == ch && al > cl);
}

// ---------------------------------------------------- block-level helpers
__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }
__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Exclusive scan over the CTA in thread order; `scratch` holds NWARP entries.
// Deterministic (integer adds); returns the CTA total in *total.
template <typename T>
__device__ __forceinline__ T block_excl_scan(T v, T* scratch, T* total) {
  const int l = lane_id(), w = warp_id();
  T incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T t = __shfl_up_sync(0xffffffffu, incl, o);
    if (l >= o) incl += t;
  }
  __syncthreads();
  if (l == 31) scratch[w] = incl;
  __syncthreads();
  T off = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < NWARP; ++i) {
    T s = scratch[i];
    if (i < w) off += s;
    tot += s;
  }
  *total = tot;
  return off + incl - v;
}

}  // namespace sv
