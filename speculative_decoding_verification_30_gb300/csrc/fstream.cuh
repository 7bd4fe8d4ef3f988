// fstream.cuh -- one-CTA-per-row verify path for sampled sequences with fp32 rows.
//
// Included by spec_verify.cu after keyhist.cuh. It shares that path's workspace
// (row results KhRow, tickets, kept-token lists, hand-back flags, work counter)
// and its per-token arithmetic (kh_w weights, kh_kept, kh_elem, fixed-point
// masses, the exact 128-bit inverse-CDF crossing test).
//
// A persistent grid of FT-thread CTAs (two per SM) takes the rows of the batch's
// sampled sequences from a work counter, sequence by sequence in the order
// fs_order_kernel wrote (heaviest sequences first). Per row, by its truncation
// parameters:
//   top-k (0 < k <= 256): the row streams through a ring of bulk copies into
//     shared memory; the k-th largest of the threads' maxima over the first two
//     stages is at most the row's k-th largest logit, so every top-k token lies at
//     or above it, and those logits are listed as composite keys (order key << 32
//     | ~id, so descending keys are logit descending, id ascending). A radix select
//     over the list finds the k-th key and ranking the candidates at or above it
//     gives the top k in order; a top-p cut falls inside them.
//   no truncation: the same ring; per-thread running sums of the weights
//     2^((z - m_t) c) with a running maximum m_t (rescaled when m_t grows).
//   top-p only: each weight 2^((z - R) c) (R = the first wave's maximum) goes to a
//     per-thread bin by its binade (shared memory, no atomics); weights 2^24 or
//     more above R are listed instead and given exact masses afterwards. The bin
//     where the exclusive mass first exceeds P * Z is read again from L2, split
//     into 256 sub-bins by the weight's top mantissa bits (exact fixed-point
//     masses) with its logits listed on the way; the crossing sub-bin's logits are
//     sorted and walked to the exact cut.
// The row's result (cut logit, id cut, 2^44 / kept mass, maximum, c) and the
// probability of the sequence's drafted token at that position go to the
// workspace. The CTA that finishes a sequence's last row runs the acceptance
// tests in order and draws the replacement from (p - q)+ or the bonus token from
// p_K by an inverse CDF in token-id order, over the listed kept tokens when the
// target row has a list, else over the whole rows (from L2).
//
// Rows this path does not serve (top-k above 256, a candidate list or crossing
// sub-bin that overflows, more than 256 weights above the bins, a crossing in the
// last bin) hand their sequence to the cluster kernel, as the bf16 path does.
#pragma once

namespace sv {

constexpr int FT = 512;                      // threads per CTA
constexpr int FWARP = FT / 32;
constexpr int FPF = 4;                       // float4 vectors per thread and load wave
constexpr int FLCAP = 4096;                  // listed candidates (u64 composite keys)
constexpr int FNB = 48;                      // coarse weight bins (one binade each)
constexpr int FB_TOP = 150;                  // bin = FB_TOP - exponent field of the weight
constexpr int FNSUB = 256;                   // sub-bins of the crossing bin
constexpr int FKMAX = 256;                   // largest top_k served here
constexpr int FOCAP = 256;                   // top-p logits above the bins (u64 composite keys)
constexpr int FRS = 4;                       // bulk-copy ring: stages
constexpr int FRV = 1024;                    // bulk-copy ring: 16-byte vectors per stage (16 KB)
constexpr int FRP = FRV / FT;                // vectors per thread and stage
constexpr int FMAXBLK = 128;                 // 32-vector blocks per warp range (V <= 262144)
constexpr size_t FS_SMEM = (size_t)FNB * FT * 4;   // bins | list | sampling block sums

struct FsShared {
  unsigned long long s64[FWARP];
  unsigned long long s64b[FWARP];
  uint32_t s32[FWARP];
  float fmax[FWARP];
  uint32_t cmax;                             // first-wave maximum (order key)
  uint32_t lcount;                           // candidates pushed
  uint32_t rflags;                           // row flags raised during the stream
  uint32_t hsel[2];                          // radix select: digit, remaining rank
  int item, last, flags, nacc, tok;
  uint32_t llen[17];
  uint32_t flag[16];
  float pz[16], qz[16];
  unsigned long long binm[FNB];
  uint32_t dh[256];                          // radix-select digit counts
  unsigned long long smass[FNSUB];           // exact masses of the crossing bin's sub-bins
  unsigned long long mabove;                 // exclusive mass before the crossing sub-bin
  int jstar, sstar, ncut;
  float zt;
  int idcut;
  unsigned long long zkept;
  unsigned long long rfull[FRS];             // bulk-copy ring: stage filled
  uint32_t rtimeout;                         // a ring wait gave up
  uint32_t ocount;                           // logits above the bins (top-p rows)
  unsigned long long olist[FOCAP];
};

#ifdef SV_TRACE
// trace builds: which hand-back a row took (bits 28..31 of its trace word)
#define FS_WHY(code)                                                                    \
  do {                                                                                  \
    if (threadIdx.x == 0 && S.item < 8192) g_khtrace[S.item * 8 + 7] |= (unsigned long long)(code) << 28; \
  } while (0)
#else
#define FS_WHY(code) \
  do {               \
  } while (0)
#endif
constexpr uint32_t FS_OVER = 8u;             // a weight beyond the bins (hand back)

// Streaming load with an L2 eviction policy: rows that are read again (a top-p
// row's refinement passes, a full-row sampling pass) stay in L2 ahead of rows
// read once.
__device__ __forceinline__ float4 fs_ld(const float4* p, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ float4 fs_ld_l2(const float4* p) { return __ldcg(p); }
// Asks L2 to fetch bytes [p, p + n) of global memory (16-byte aligned, n a
// multiple of 16), in 32 KB pieces spread over the calling warp's lanes.
__device__ __forceinline__ void fs_prefetch_l2(const void* p, size_t n) {
  const char* c = static_cast<const char*>(p);
  for (size_t off = (size_t)lane_id() * 32768u; off < n; off += 32u * 32768u) {
    const uint32_t sz = (uint32_t)min((size_t)32768u, n - off);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c + off), "r"(sz) : "memory");
  }
}

__device__ __forceinline__ float fs_at(const float4& v, int e) {
  return e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
}
// y = (z - R) c, the log2 weight of logit z against the reference R: formed as a
// difference then a product (not z c - R c), so that a large |R c| adds no
// rounding error; every pass over a row uses this one formula.
__device__ __forceinline__ float fs_y(float z, float R, float c) { return __fmul_rn(__fsub_rn(z, R), c); }
// Coarse bin of a weight w = 2^y (y = (z - R) c relative to the first-wave
// maximum R), from w's exponent field: bin j holds w in [2^(23 - j), 2^(24 - j)),
// a negative value is above the bins (w >= 2^24), and everything below the last
// bin's binade joins that bin. Both passes over a row bin by this one formula.
__device__ __forceinline__ int fs_bin_of(float w) { return FB_TOP - (int)(__float_as_uint(w) >> 23); }

// Warp 0 of a radix select: the digit (255 down to 0) whose count in S.dh holds
// the kk-th largest key, and the rank left inside it, into S.hsel. Lane l holds
// digits 255 - 8l down to 248 - 8l.
__device__ __forceinline__ void fs_pick_digit(uint32_t kk, FsShared& S) {
  const int l = lane_id();
  uint32_t c8[8], s = 0u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c8[j] = S.dh[255 - 8 * l - j];
    s += c8[j];
  }
  uint32_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (l >= o) incl += t;
  }
  const uint32_t excl = incl - s;
  if (excl < kk && kk <= incl) {
    uint32_t run = excl;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (run + c8[j] >= kk) {
        S.hsel[0] = (uint32_t)(255 - 8 * l - j);
        S.hsel[1] = kk - run;
        break;
      }
      run += c8[j];
    }
  }
}

// k-th largest (1-based, k <= FT) of the CTA's per-thread 32-bit keys, by four
// rounds of 8-bit digits (most significant first). Every thread returns it.
__device__ __noinline__ uint32_t fs_kth_key(uint32_t key, int k, FsShared& S) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0u, pmask = 0u;
  uint32_t kk = (uint32_t)k;
  for (int r = 0; r < 4; ++r) {
    const int sh = 24 - 8 * r;
    for (int i = tid; i < 256; i += FT) S.dh[i] = 0u;
    __syncthreads();
    if ((key & pmask) == prefix) atomicAdd(&S.dh[(key >> sh) & 255u], 1u);
    __syncthreads();
    if (tid < 32) fs_pick_digit(kk, S);
    __syncthreads();
    prefix |= S.hsel[0] << sh;
    pmask |= 255u << sh;
    kk = S.hsel[1];
    __syncthreads();
  }
  return prefix;
}

// Value key (upper 32 bits) of the k-th largest of the n composites a[0, n)
// (k <= n), by four rounds of 8-bit digits over the list. Every thread returns it.
__device__ __noinline__ uint32_t fs_kth_listed(const unsigned long long* a, int n, int k, FsShared& S) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0u, pmask = 0u;
  uint32_t kk = (uint32_t)k;
  for (int r = 0; r < 4; ++r) {
    const int sh = 24 - 8 * r;
    __syncthreads();
    for (int i = tid; i < 256; i += FT) S.dh[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += FT) {
      const uint32_t key = (uint32_t)(a[i] >> 32);
      if ((key & pmask) == prefix) atomicAdd(&S.dh[(key >> sh) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) fs_pick_digit(kk, S);
    __syncthreads();
    prefix |= S.hsel[0] << sh;
    pmask |= 255u << sh;
    kk = S.hsel[1];
  }
  __syncthreads();
  return prefix;
}

// Sorts a[0, n) descending in place (n a power of two, entries past the data 0).
__device__ __noinline__ void fs_sort_desc(unsigned long long* a, int n) {
  __syncthreads();
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n / 2; i += FT) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long x = a[lo], y = a[hi];
        if (desc ? x < y : x > y) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

__device__ __forceinline__ float fs_key_value(unsigned long long e) { return key_to_float((uint32_t)(e >> 32)); }
__device__ __forceinline__ int fs_key_id(unsigned long long e) { return (int)~(uint32_t)e; }

// Pushes the logits of vector v that are >= thr as composite keys (one atomic per
// vector with candidates; nothing is written past FLCAP).
__device__ __forceinline__ void fs_push(const float4& x, int v, float thr, FsShared& S,
                                        unsigned long long* list) {
  uint32_t mk = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) mk |= (uint32_t)(fs_at(x, e) >= thr) << e;
  if (!mk) return;
  uint32_t slot = atomicAdd(&S.lcount, (uint32_t)__popc(mk));
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (!((mk >> e) & 1u)) continue;
    if (slot < (uint32_t)FLCAP)
      list[slot] = ((unsigned long long)okey(fs_at(x, e)) << 32) | (uint32_t)~(uint32_t)(4 * v + e);
    ++slot;
  }
}

// Row classes.
constexpr int FC_TOPK = 0, FC_ALL = 1, FC_TOPP = 2;

// Lists the logits of vector v whose weight 2^((z - R) c) lies above the bins
// (2^24 or more times the first-wave maximum's): their masses are taken exactly
// after the stream. Sets *over when the list is full.
__device__ __noinline__ void fs_push_over(float4 x, int v, float c, float R, FsShared& S,
                                          uint32_t* over) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float z = fs_at(x, e);
    if (fs_bin_of(ex2_approx(fs_y(z, R, c))) >= 0) continue;
    const uint32_t slot = atomicAdd(&S.ocount, 1u);
    if (slot < (uint32_t)FOCAP)
      S.olist[slot] = ((unsigned long long)okey(z) << 32) | (uint32_t)~(uint32_t)(4 * v + e);
    else
      *over = 1u;
  }
}

// One pass over a top-p row (double-buffered waves of FPF vectors per thread in
// registers: the bins fill the shared memory). Returns this thread's maximum and
// the first wave's block maximum R in *Rout; *nan is set on NaN or +inf. Each
// weight 2^((z - R) c) is added to the thread's bin of its binade; weights above
// the bins are listed (S.olist), and more than FOCAP of them raise FS_OVER.
__device__ __noinline__ float fs_stream_topp(const float4* src, int nv, float c, FsShared& S, float* bins,
                                             float* Rout, bool* nan) {
  const int tid = threadIdx.x, l = lane_id();
  // read again by the refinement passes: kept in L2 ahead of rows read once
  const uint64_t pol = policy_evict_last();
  float4 cur[FPF], nxt[FPF];
  const float4 NEG = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
  for (int p = 0; p < FPF; ++p) {
    const int q = tid + p * FT;
    cur[p] = q < nv ? fs_ld(src + q, pol) : NEG;
  }
  float tmax = -INFINITY;
  bool bad = false;
#pragma unroll
  for (int p = 0; p < FPF; ++p)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float z = fs_at(cur[p], e);
      tmax = fmaxf(tmax, z);
      bad |= !(z == z) || z == INFINITY;
    }
  // the second wave is in flight while the block agrees on R
#pragma unroll
  for (int p = 0; p < FPF; ++p) {
    const int q = tid + FPF * FT + p * FT;
    nxt[p] = q < nv ? fs_ld(src + q, pol) : NEG;
  }
  float fm = tmax;
#pragma unroll
  for (int o = 16; o; o >>= 1) fm = fmaxf(fm, __shfl_xor_sync(0xffffffffu, fm, o));
  __syncthreads();
  if (tid == 0) {
    S.cmax = okey(-INFINITY);
    S.lcount = 0u;
    S.rflags = 0u;
    S.ocount = 0u;
    S.rtimeout = 0u;
  }
  __syncthreads();
  if (l == 0) atomicMax(&S.cmax, okey(fm));
  __syncthreads();
  const float R = key_to_float(S.cmax);
  *Rout = R;
  uint32_t over = 0u;
  for (int q0 = tid; q0 < nv; q0 += FPF * FT) {
#pragma unroll
    for (int p = 0; p < FPF; ++p) {
      const int q = q0 + p * FT;
      if (q >= nv) continue;
      const float4 x = cur[p];
      const float vm = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
      tmax = fmaxf(tmax, vm);
      bad |= !(x.x == x.x) || !(x.y == x.y) || !(x.z == x.z) || !(x.w == x.w) || vm == INFINITY;
      bool ov = false;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float w = ex2_approx(fs_y(fs_at(x, e), R, c));
        const int bb = fs_bin_of(w);
        ov |= bb < 0;
        bins[min(max(bb, 0), FNB - 1) * FT + tid] += bb >= 0 ? w : 0.0f;
      }
      if (ov) fs_push_over(x, q, c, R, S, &over);
    }
#pragma unroll
    for (int p = 0; p < FPF; ++p) cur[p] = nxt[p];
#pragma unroll
    for (int p = 0; p < FPF; ++p) {
      const int q = q0 + 2 * FPF * FT + p * FT;
      nxt[p] = q < nv ? fs_ld(src + q, pol) : NEG;
    }
  }
  if (over) atomicOr(&S.rflags, FS_OVER);
  *nan = bad;
  return tmax;
}

// One pass over a top-k or untruncated row through a ring of FRS shared-memory
// stages of 16 KB, filled by bulk copies (one thread issues them; FRS - 1 stages
// stay in flight while the CTA reads one), so that a CTA keeps 48 KB of the row in
// flight without registers. Returns the thread maximum, with the first two
// stages' block maximum R; top-k rows list the logits at or above the k-th
// largest thread maximum of those stages, untruncated rows leave the thread's
// running (max, sum) in *mt / *st.
// Every wait is bounded; on a timeout the row is marked (S.rtimeout) after the
// copies in flight have landed.
template <int CLS>
__device__ __noinline__ float fs_stream_ring(const float4* src, int nv, int k, float c, FsShared& S,
                                             unsigned long long* list, float4* ring, float* mt,
                                             float* st, float* Rout, bool* nan) {
  const int tid = threadIdx.x, l = lane_id();
  const int nst = (nv + FRV - 1) / FRV;
  const uint64_t pol = CLS == FC_TOPK ? policy_evict_first() : policy_evict_last();
  // the previous row's writes to this shared memory come before the bulk copies
  fence_proxy_async();
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < FRS; ++s) mbar_init(&S.rfull[s], 1);
    fence_mbar_init();
    S.cmax = okey(-INFINITY);
    S.lcount = 0u;
    S.rflags = 0u;
    S.ocount = 0u;
    S.rtimeout = 0u;
  }
  __syncthreads();
  int issued = min(FRS, nst);                  // stages issued (thread 0's count)
  if (tid == 0) {
    for (int s = 0; s < issued; ++s) {
      const uint32_t bytes = (uint32_t)min(FRV, nv - s * FRV) * 16u;
      mbar_arrive_expect_tx(&S.rfull[s], bytes);
      bulk_g2s(ring + (size_t)s * FRV, src + (size_t)s * FRV, bytes, &S.rfull[s], pol);
    }
  }
  bool tmo = false;
  // first two stages (16 logits per thread): block maximum R, top-k threshold
  float tmax = -INFINITY;
  bool bad = false;
  for (int s = 0; s < 2 && s < nst; ++s) {
    if (!mbar_wait_bounded(&S.rfull[s], 0u, WAIT_LIMIT_NS)) tmo = true;
#pragma unroll
    for (int p = 0; p < FRP; ++p) {
      const int q = s * FRV + tid + p * FT;
      if (q >= nv) continue;
      const float4 x = ring[(size_t)s * FRV + tid + p * FT];
      tmax = fmaxf(tmax, fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)));
    }
  }
  float fm = tmax;
#pragma unroll
  for (int o = 16; o; o >>= 1) fm = fmaxf(fm, __shfl_xor_sync(0xffffffffu, fm, o));
  if (l == 0) atomicMax(&S.cmax, okey(fm));
  __syncthreads();
  const float R = key_to_float(S.cmax);
  *Rout = R;
  float th = -INFINITY;
  if (CLS == FC_TOPK) th = key_to_float(fs_kth_key(okey(tmax), k, S));
  float m_t = -INFINITY, s_t = 0.0f;
  for (int s = 0; s < nst; ++s) {
    const int slot = s % FRS;
    if (s >= 2 && !mbar_wait_bounded(&S.rfull[slot], (uint32_t)((s / FRS) & 1), WAIT_LIMIT_NS)) tmo = true;
    if (!tmo) {
#pragma unroll
      for (int p = 0; p < FRP; ++p) {
        const int q = s * FRV + tid + p * FT;
        if (q >= nv) continue;
        const float4 x = ring[(size_t)slot * FRV + tid + p * FT];
        const float vm = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
        tmax = fmaxf(tmax, vm);
        bad |= !(x.x == x.x) || !(x.y == x.y) || !(x.z == x.z) || !(x.w == x.w) || vm == INFINITY;
        if (CLS == FC_TOPK) {
          if (vm >= th) fs_push(x, q, th, S, list);
        } else {
          if (vm > m_t) {
            s_t = m_t > -INFINITY ? s_t * ex2_approx((m_t - vm) * c) : 0.0f;
            m_t = vm;
          }
          s_t += (ex2_approx(fs_y(x.x, m_t, c)) + ex2_approx(fs_y(x.y, m_t, c))) +
                 (ex2_approx(fs_y(x.z, m_t, c)) + ex2_approx(fs_y(x.w, m_t, c)));
        }
      }
    }
    // the stage is read by every thread before it is filled again
    if (__syncthreads_or(tmo ? 1 : 0)) {
      tmo = true;
      break;
    }
    if (tid == 0 && s + FRS < nst) {
      const uint32_t bytes = (uint32_t)min(FRV, nv - (s + FRS) * FRV) * 16u;
      mbar_arrive_expect_tx(&S.rfull[slot], bytes);
      bulk_g2s(ring + (size_t)slot * FRV, src + (size_t)(s + FRS) * FRV, bytes, &S.rfull[slot], pol);
      ++issued;
    }
  }
  if (tmo) {
    // let every copy this row issued land before the ring is reused
    if (tid == 0) {
      S.rtimeout = 1u;
      for (int s = max(0, issued - FRS); s < issued; ++s)
        mbar_wait_bounded(&S.rfull[s % FRS], (uint32_t)((s / FRS) & 1), WAIT_LIMIT_NS);
    }
    __syncthreads();
  }
  *mt = m_t;
  *st = s_t;
  *nan = bad;
  return tmax;
}

// Second and third passes of a top-p row (from L2): sub-bin histogram of coarse
// bin j with the bin's logits listed (PASS 2), or the list of sub-bin s of bin j
// (PASS 3). List slots are taken per warp; nothing is written past FLCAP.
template <int PASS>
__device__ __noinline__ void fs_refine(const float4* src, int nv, float c, float R, float scale, int j,
                                       int s, FsShared& S, unsigned long long* list) {
  const int tid = threadIdx.x, l = lane_id();
  const uint32_t below = (1u << l) - 1u;
  const float ylo = (float)(22 - j) + 0.99f, yhi = (float)(24 - j) + 0.01f;
  float4 cur[FPF], nxt[FPF];
  const float4 NEG = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
  for (int p = 0; p < FPF; ++p) {
    const int q = tid + p * FT;
    cur[p] = q < nv ? fs_ld_l2(src + q) : NEG;
  }
  // warp-uniform trip count (the ballots below need every lane)
  for (int qb = tid - l; qb < nv; qb += FPF * FT) {
    const int q0 = qb + l;
#pragma unroll
    for (int p = 0; p < FPF; ++p) {
      const int q = q0 + FPF * FT + p * FT;
      nxt[p] = q < nv ? fs_ld_l2(src + q) : NEG;
    }
#pragma unroll
    for (int p = 0; p < FPF; ++p) {
      const int q = q0 + p * FT;
      // bin j < FNB - 1 exactly (the listed logits above the bins excluded); the
      // weight is formed only for logits whose y lies within 0.01 of the bin's
      // binade (ex2's rounding moves a weight across a binade only within ~1e-6)
      uint32_t m4 = 0u;
      float w4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float y = fs_y(fs_at(cur[p], e), R, c);
        w4[e] = 0.0f;
        if (q < nv && y >= ylo && y < yhi) {
          w4[e] = ex2_approx(y);
          m4 |= (uint32_t)(fs_bin_of(w4[e]) == j) << e;
        }
      }
      if (!__any_sync(0xffffffffu, m4 != 0u)) continue;
      const bool lfull = PASS == 2 && *reinterpret_cast<volatile uint32_t*>(&S.lcount) > (uint32_t)FLCAP;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float z = fs_at(cur[p], e);
        const bool inb = (m4 >> e) & 1u;
        const float w = w4[e];
        const int sb = (int)((__float_as_uint(w) >> 15) & 255u);
        if (PASS == 2 && inb) atomicAdd(&S.smass[sb], fix_pow2(w * scale, FIX));
        // (pass 2 stops listing once the bin has overflowed the list: pass 3 runs)
        const bool want = PASS == 2 ? inb && !lfull : (inb && sb == s);
        const uint32_t mk = __ballot_sync(0xffffffffu, want);
        if (mk) {
          const int ld = __ffs(mk) - 1;
          uint32_t base = 0u;
          if (l == ld) base = atomicAdd(&S.lcount, (uint32_t)__popc(mk));
          base = __shfl_sync(0xffffffffu, base, ld);
          const uint32_t slot = base + (uint32_t)__popc(mk & below);
          if (want && slot < (uint32_t)FLCAP)
            list[slot] = ((unsigned long long)okey(z) << 32) | (uint32_t)~(uint32_t)(4 * q + e);
        }
      }
    }
#pragma unroll
    for (int p = 0; p < FPF; ++p) cur[p] = nxt[p];
  }
}

__device__ __forceinline__ int fs_pow2(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

// One fp32 row: stream, cut, normaliser, and the probability of the drafted token
// d (-1: none). Top-k rows list their kept tokens in glist (ids, no order). The
// result is returned in every thread; pad[0] holds p(d) as float bits, pad[1] the
// list length or KH_NOLIST.
__device__ __noinline__ KhRow fs_row(const float* row, int V, float T, int k, float topP, int d,
                                     uint32_t* glist, FsShared& S) {
  const int tid = threadIdx.x, l = lane_id(), w = warp_id();
  const int nv = V / 4;
  const float4* src = reinterpret_cast<const float4*>(row);
  const float c = __fdiv_rn(KH_LOG2E, T);
  const bool topk = k > 0 && k < V;
  const bool topp = topP < 1.0f;
  const int cls = topk ? FC_TOPK : (topp ? FC_TOPP : FC_ALL);
  unsigned long long* list = reinterpret_cast<unsigned long long*>(kh_dyn);
  float* bins = reinterpret_cast<float*>(kh_dyn);
  KhRow res;
  res.c = c;
  res.zt = -INFINITY;
  res.idcut = V;
  res.invZ = 0.0f;
  res.flags = 0u;
  res.pad[0] = 0u;
  res.pad[1] = KH_NOLIST;
  if (topk && k > FKMAX) {
    res.m = 0.0f;
    res.flags = KH_BAIL;
    FS_WHY(1);
    return res;
  }
  if (cls == FC_TOPP) {
    __syncthreads();
    for (int j = 0; j < FNB; ++j) bins[j * FT + tid] = 0.0f;
    __syncthreads();
  }
  float mt, st, R;
  bool nan;
  float tm;
  // top-k and untruncated rows stream through a bulk-copy ring placed after the
  // candidate list (its first FLCAP entries)
  float4* ring = reinterpret_cast<float4*>(list + FLCAP);
  if (cls == FC_TOPK) tm = fs_stream_ring<FC_TOPK>(src, nv, k, c, S, list, ring, &mt, &st, &R, &nan);
  else if (cls == FC_ALL) tm = fs_stream_ring<FC_ALL>(src, nv, k, c, S, list, ring, &mt, &st, &R, &nan);
  else tm = fs_stream_topp(src, nv, c, S, bins, &R, &nan);
#pragma unroll
  for (int o = 16; o; o >>= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
  if (l == 0) S.fmax[w] = tm;
  const bool anynan = __syncthreads_or(nan ? 1 : 0) != 0;
  float m = S.fmax[0];
#pragma unroll
  for (int i = 1; i < KWARP; ++i) m = fmaxf(m, S.fmax[i]);
  res.m = m;
  KH_MARK(S.item, 1);
  if (anynan || !(m > -INFINITY) || S.rtimeout) {
    res.flags = KH_ERR;
    return res;
  }
  if (S.rflags & FS_OVER) {
    res.flags = KH_BAIL;
    FS_WHY(2);
    return res;
  }
  unsigned long long Zk = 0ull;
  if (cls == FC_ALL) {
    // sum of the threads' running sums, each moved to the frame of m
    unsigned long long t = mt > -INFINITY ? fix_pow2(st * ex2_approx((mt - m) * c), FIX) : 0ull;
    t = warp_sum(t);
    __syncthreads();
    if (l == 0) S.s64[w] = t;
    __syncthreads();
    for (int i = 0; i < KWARP; ++i) Zk += S.s64[i];
  } else if (cls == FC_TOPK) {
    const uint32_t nl = S.lcount;
    if (nl > (uint32_t)FLCAP || nl < (uint32_t)k) {
      res.flags = KH_BAIL;
      FS_WHY(3);
      return res;
    }
    // the k-th largest logit key; the candidates at or above it (the top k plus any
    // further ties of that key) ranked by composite key: rank < k is the top k
    const uint32_t kth = fs_kth_listed(list, (int)nl, k, S);
    KH_MARK(S.item, 2);
    unsigned long long* cand = list + FLCAP;
    if (tid == 0) S.ncut = 0;
    __syncthreads();
    for (int i = tid; i < (int)nl; i += FT) {
      const unsigned long long e = list[i];
      if ((uint32_t)(e >> 32) >= kth) {
        const uint32_t slot = atomicAdd((uint32_t*)&S.ncut, 1u);
        if (slot < (uint32_t)FLCAP) cand[slot] = e;
      }
    }
    __syncthreads();
    const int nc = S.ncut;
    if (nc > FLCAP) {
      res.flags = KH_BAIL;
      FS_WHY(4);
      return res;
    }
    if (nc <= 1024) {
      // rank by counting (composite keys are distinct)
      for (int i = tid; i < nc; i += FT) {
        const unsigned long long e = cand[i];
        int rank = 0;
        for (int j = 0; j < nc; ++j) rank += (int)(cand[j] > e);
        if (rank < k) list[rank] = e;
      }
    } else {
      // many ties of the k-th key: sort the candidates
      const int n2 = fs_pow2(nc);
      for (int i = nc + tid; i < n2; i += FT) cand[i] = 0ull;
      fs_sort_desc(cand, n2);
      for (int i = tid; i < k; i += FT) list[i] = cand[i];
    }
    __syncthreads();
    // the top k in order; their exact fixed-point weights and exclusive sums
    unsigned long long wk = 0ull;
    if (tid < k) wk = fix_pow2(kh_w(fs_key_value(list[tid]), m, c), FIX);
    unsigned long long ZL1;
    const unsigned long long ex = kh_below<unsigned long long>(wk, S.s64, &ZL1);
    int nkeep = k;
    if (topp) {
      const unsigned long long Y = mass_threshold(topP, ZL1);
      // kept iff the exclusive mass <= Y: a prefix of the k entries
      nkeep = __syncthreads_count(tid < k && ex <= Y);
    }
    if (tid == nkeep - 1) {
      S.zt = fs_key_value(list[tid]);
      S.idcut = fs_key_id(list[tid]);
      S.zkept = ex + wk;
    }
    if (glist)
      for (int i = tid; i < nkeep; i += FT) glist[i] = (uint32_t)fs_key_id(list[i]);
    __syncthreads();
    res.zt = S.zt;
    res.idcut = S.idcut;
    res.pad[1] = (uint32_t)nkeep;
    Zk = S.zkept;
  } else {
    // top-p: bin masses in the frame of m; warp w sums bins w and w + 16
    const float scale = ex2_approx((R - m) * c);
    for (int j = w; j < FNB; j += KWARP) {
      unsigned long long t = 0ull;
      for (int i = l; i < FT; i += 32) t += fix_pow2(bins[j * FT + i] * scale, FIX);
      t = warp_sum(t);
      if (l == 0) S.binm[j] = t;
    }
    __syncthreads();
    // the logits above the bins, sorted, with exact masses in the frame of m
    const int no = (int)S.ocount;            // <= FOCAP (more were handed back)
    unsigned long long om = 0ull;
    if (no > 0) {
      const int n2 = fs_pow2(no);
      for (int i = no + tid; i < n2; i += FT) S.olist[i] = 0ull;
      fs_sort_desc(S.olist, n2);
      if (tid < no) om = fix_pow2(kh_w(fs_key_value(S.olist[tid]), m, c), FIX);
    }
    unsigned long long OZ;
    const unsigned long long oex = kh_below<unsigned long long>(om, S.s64, &OZ);
    unsigned long long Z = OZ;
    for (int j = 0; j < FNB; ++j) Z += S.binm[j];
    const unsigned long long Y = mass_threshold(topP, Z);
    if (OZ > Y) {
      // the cut lies among them: kept while the exclusive mass is <= Y
      const int nk = __syncthreads_count(tid < no && oex <= Y);
      if (tid == nk - 1) {
        S.zt = fs_key_value(S.olist[tid]);
        S.idcut = fs_key_id(S.olist[tid]);
        S.zkept = oex + om;
      }
      __syncthreads();
      res.zt = S.zt;
      res.idcut = S.idcut;
      Zk = S.zkept;
    } else {
      // the bin where the exclusive mass first exceeds Y
      int js = -1;
      unsigned long long above = OZ;
      for (int j = 0; j < FNB; ++j) {
        if (above + S.binm[j] > Y) {
          js = j;
          break;
        }
        above += S.binm[j];
      }
      if (js < 0 || js == FNB - 1) {
        res.flags = KH_BAIL;
        FS_WHY(5);
        return res;
      }
      // sub-bins of bin js (exact masses) from L2; the bin's logits listed
      __syncthreads();
      for (int i = tid; i < FNSUB; i += FT) S.smass[i] = 0ull;
      if (tid == 0) S.lcount = 0u;
      __syncthreads();
      fs_refine<2>(src, nv, c, R, scale, js, 0, S, list);
      __syncthreads();
      KH_MARK(S.item, 2);
      if (tid == 0) {
        int ss = -1;
        unsigned long long cum = above;
        for (int sb = FNSUB - 1; sb >= 0; --sb) {
          const unsigned long long sm = S.smass[sb];
          if (cum + sm > Y) {
            ss = sb;
            break;
          }
          cum += sm;
        }
        S.sstar = ss;
        S.mabove = cum;
        S.ncut = 0;
      }
      __syncthreads();
      const int ss = S.sstar;
      if (ss < 0) {
        res.flags = KH_BAIL;                   // rounding left the crossing outside the bin
        FS_WHY(6);
        return res;
      }
      const uint32_t nbin = S.lcount;
      uint32_t nl;
      unsigned long long* sel = list;
      if (nbin <= (uint32_t)FLCAP) {
        // the crossing sub-bin's entries of the listed bin
        sel = list + FLCAP;
        for (int i = tid; i < (int)nbin; i += FT) {
          const unsigned long long e = list[i];
          const float wv = ex2_approx(fs_y(fs_key_value(e), R, c));
          if ((int)((__float_as_uint(wv) >> 15) & 255u) == ss) sel[atomicAdd((uint32_t*)&S.ncut, 1u)] = e;
        }
        __syncthreads();
        nl = (uint32_t)S.ncut;
      } else {
        // too many to list: list the crossing sub-bin in a third pass
        __syncthreads();
        if (tid == 0) S.lcount = 0u;
        __syncthreads();
        fs_refine<3>(src, nv, c, R, scale, js, ss, S, list);
        __syncthreads();
        nl = S.lcount;
      }
      if (nl > (uint32_t)FLCAP || nl == 0u) {
        res.flags = KH_BAIL;
        FS_WHY(7);
        return res;
      }
      const int n2 = fs_pow2((int)nl);
      for (int i = (int)nl + tid; i < n2; i += FT) sel[i] = 0ull;
      fs_sort_desc(sel, n2);
      list = sel;
      KH_MARK(S.item, 3);
      // the sorted entries are kept while their exclusive mass is <= Y (a prefix, at
      // least the first entry); their weights as the sub-bin masses summed them.
      // Thread t takes entries [t e, t e + e) in order; a scan gives its offset.
      const int ept = ((int)nl + FT - 1) / FT;
      const int i0 = min(tid * ept, (int)nl), i1 = min(i0 + ept, (int)nl);
      unsigned long long own = 0ull;
      for (int i = i0; i < i1; ++i) own += fix_pow2(ex2_approx(fs_y(fs_key_value(list[i]), R, c)) * scale, FIX);
      if (tid == 0) S.jstar = 0;
      unsigned long long wtot;
      unsigned long long ex = S.mabove + kh_below<unsigned long long>(own, S.s64, &wtot);
      int lastk = -1;
      unsigned long long zk = 0ull;
      for (int i = i0; i < i1; ++i) {
        if (ex > Y) break;
        lastk = i;
        ex += fix_pow2(ex2_approx(fs_y(fs_key_value(list[i]), R, c)) * scale, FIX);
        zk = ex;
      }
      if (lastk > 0) atomicMax(&S.jstar, lastk);
      __syncthreads();
      const int last = S.jstar;
      if (lastk == last) {
        S.zt = fs_key_value(list[last]);
        S.idcut = fs_key_id(list[last]);
        S.zkept = zk;
      }
      __syncthreads();
      res.zt = S.zt;
      res.idcut = S.idcut;
      Zk = S.zkept;
    }
  }
  if (Zk == 0ull) {
    res.flags = KH_BAIL;
    FS_WHY(8);
    return res;
  }
  res.invZ = __fdiv_rn(17592186044416.0f, (float)Zk);   // 2^44 / Z
  if (d >= 0) {
    const float zd = __ldg(row + d);
    const float pd = kh_kept(zd, d, res.zt, res.idcut) ? __fmul_rn(kh_w(zd, m, c), res.invZ) : 0.0f;
    res.pad[0] = __float_as_uint(pd);
  }
  return res;
}

// Fixed-point (2^-40) mass of the 4 tokens of vector v: the residual (p - q)+
// (RES; target logits a, draft logits b) or the target probability p.
template <bool RES>
__device__ __forceinline__ unsigned long long fs_vec_mass(const float4& a, const float4& b, int v, const KhW& tp,
                                                          const KhW& tq) {
  unsigned long long acc = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float r, p;
    kh_elem(fs_at(a, e), fs_at(b, e), 4 * v + e, RES, tp, tq, &r, &p);
    acc += fixr(RES ? r : p);
  }
  return acc;
}

// One inverse-CDF pass over whole fp32 rows (from L2) for the residual (RES) or
// the target p: the smallest id j whose running mass S_j satisfies
// S_j * 2^24 > kv * S (S the total). Warps sum contiguous ranges per 32-vector
// block; warp 0 locates the crossing block with lane-parallel scans and walks it.
// -1 if no token qualifies, -2 if the total mass is 0.
template <bool RES>
__device__ __noinline__ int fs_sample_pass(const float4* sp, const float4* sq, int nv, KhW tp, KhW tq, uint32_t kv,
                                           FsShared& S) {
  const int w = warp_id(), l = lane_id();
  const int cw = (nv + FWARP - 1) / FWARP;
  const int nb = (cw + 31) / 32;
  const int a0 = min(w * cw, nv), a1 = min(a0 + cw, nv);
  unsigned long long* bm = reinterpret_cast<unsigned long long*>(kh_dyn);
  const float4 NEG = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  unsigned long long tot = 0;
  constexpr int U = 4;                         // blocks whose vectors are in flight at once
  for (int j0 = 0; j0 < nb; j0 += U) {
    float4 av[U], bv4[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = a0 + (j0 + u) * 32 + l;
      const bool in = j0 + u < nb && v < a1;
      av[u] = in ? __ldcg(sp + v) : NEG;
      bv4[u] = in && RES ? __ldcg(sq + v) : NEG;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (j0 + u >= nb) break;
      const int v = a0 + (j0 + u) * 32 + l;
      unsigned long long x = v < a1 ? fs_vec_mass<RES>(av[u], bv4[u], v, tp, tq) : 0ull;
      x = kh_wsum(x);
      if (l == 0) bm[w * FMAXBLK + j0 + u] = x;
      tot += x;
    }
  }
  __syncthreads();
  if (l == 0) S.s64[w] = tot;
  __syncthreads();
  if (w == 0) {
    const unsigned long long own = l < FWARP ? S.s64[l] : 0ull;
    const unsigned long long St = warp_sum(own);
    unsigned long long incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
      if (l >= o) incl += t;
    }
    const uint32_t bw = __ballot_sync(0xffffffffu, l < FWARP && mul_gt(incl, 1ull << 24, kv, St));
    int tok = St == 0ull ? -2 : -1;
    if (St != 0ull && bw) {
      const int ww = __ffs(bw) - 1;
      unsigned long long acc = __shfl_sync(0xffffffffu, incl - own, ww);
      const int wa0 = min(ww * cw, nv), wa1 = min(wa0 + cw, nv);
      // blocks of warp ww: lane l holds blocks 4l .. 4l+3
      unsigned long long b4[4], bs = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        b4[u] = 4 * l + u < nb ? bm[ww * FMAXBLK + 4 * l + u] : 0ull;
        bs += b4[u];
      }
      unsigned long long bi = bs;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, bi, o);
        if (l >= o) bi += t;
      }
      const uint32_t bl = __ballot_sync(0xffffffffu, mul_gt(acc + bi, 1ull << 24, kv, St));
      if (bl) {
        const int lb = __ffs(bl) - 1;
        acc += __shfl_sync(0xffffffffu, bi - bs, lb);
        int jb = 4 * lb;
#pragma unroll
        for (int u = 0; u < 3; ++u) {
          const unsigned long long bu = __shfl_sync(0xffffffffu, b4[u], lb);
          if (jb == 4 * lb + u && !mul_gt(acc + bu, 1ull << 24, kv, St)) {
            acc += bu;
            ++jb;
          }
        }
        // the block: one vector per lane, in id order
        const int v = wa0 + jb * 32 + l;
        float4 a = NEG, bq = NEG;
        if (v < wa1) {
          a = __ldcg(sp + v);
          if (RES) bq = __ldcg(sq + v);
        }
        const unsigned long long mine = v < wa1 ? fs_vec_mass<RES>(a, bq, v, tp, tq) : 0ull;
        unsigned long long ci = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned long long t = __shfl_up_sync(0xffffffffu, ci, o);
          if (l >= o) ci += t;
        }
        const uint32_t hit = __ballot_sync(0xffffffffu, v < wa1 && mul_gt(acc + ci, 1ull << 24, kv, St));
        if (hit && l == __ffs(hit) - 1) {
          unsigned long long run = acc + ci - mine;
          for (int e = 0; e < 4 && tok < 0; ++e) {
            float rr, pp;
            kh_elem(fs_at(a, e), fs_at(bq, e), 4 * v + e, RES, tp, tq, &rr, &pp);
            run += fixr(RES ? rr : pp);
            if (mul_gt(run, 1ull << 24, kv, St)) tok = 4 * v + e;
          }
        }
        tok = __reduce_max_sync(0xffffffffu, tok);
      }
    }
    if (l == 0) S.tok = tok;
  }
  __syncthreads();
  return S.tok;
}

// Inverse CDF in token-id order over (p - q)+ (paired) or p, over whole fp32 rows:
// when the residual mass is 0 the target p is used. -1 if no token qualifies.
__device__ __noinline__ int fs_sample_full(const float4* sp, const float4* sq, int nv, bool paired, KhW tp,
                                           KhW tq, uint32_t kv, FsShared& S) {
  if (warp_id() == 0) {
    // both rows were streamed a while ago: fetch them back at full width
    fs_prefetch_l2(sp, (size_t)nv * 16u);
    if (paired) fs_prefetch_l2(sq, (size_t)nv * 16u);
  }
  int tok = paired ? fs_sample_pass<true>(sp, sq, nv, tp, tq, kv, S) : -2;
  if (tok == -2) tok = fs_sample_pass<false>(sp, sq, nv, tp, tq, kv, S);
  return tok < 0 ? -1 : tok;
}

// The inverse CDF of fs_sample_full over a target row whose kept tokens are
// listed (L <= 256 ids, any order): only those carry p > 0, so the sums run over
// the list sorted by id.
__device__ __noinline__ int fs_sample_list(const float* zp_row, const float* zq_row, const uint32_t* glist,
                                           int L, bool paired, KhW tp, KhW tq, uint32_t kv, FsShared& S) {
  const int tid = threadIdx.x;
  uint32_t* ids = kh_dyn;                                          // [FKMAX]
  unsigned long long* wr = reinterpret_cast<unsigned long long*>(kh_dyn + FKMAX);   // sorted r
  unsigned long long* wp = wr + FKMAX;                             // sorted p
  uint32_t* sid = reinterpret_cast<uint32_t*>(wp + FKMAX);         // sorted ids
  for (int e = tid; e < L; e += FT) ids[e] = __ldcg(glist + e);
  __syncthreads();
  for (int e = tid; e < L; e += FT) {
    const int id = (int)ids[e];
    const float zp = __ldcg(zp_row + id);
    const float zq = paired ? __ldcg(zq_row + id) : 0.0f;
    float r, p;
    kh_elem(zp, zq, id, paired, tp, tq, &r, &p);
    int rank = 0;
    for (int f = 0; f < L; ++f) rank += (int)(ids[f] < (uint32_t)id);
    wr[rank] = fixr(r);
    wp[rank] = fixr(p);
    sid[rank] = (uint32_t)id;
  }
  __syncthreads();
  const unsigned long long r1 = tid < L ? wr[tid] : 0ull, p1 = tid < L ? wp[tid] : 0ull;
  unsigned long long SR, SP;
  const unsigned long long xr = kh_below<unsigned long long>(r1, S.s64, &SR);
  const unsigned long long xp = kh_below<unsigned long long>(p1, S.s64b, &SP);
  const bool useR = SR > 0ull;
  const unsigned long long St = useR ? SR : SP;
  if (tid == 0) S.tok = -1;
  __syncthreads();
  const unsigned long long run = useR ? xr : xp, own = useR ? r1 : p1;
  if (tid < L && !mul_gt(run, 1ull << 24, kv, St) && mul_gt(run + own, 1ull << 24, kv, St)) S.tok = (int)sid[tid];
  __syncthreads();
  return S.tok;
}

// Clears sequence b's kept-token lists (their lengths are in S.llen).
__device__ __noinline__ void fs_clear_lists(const Params& P, int b, const FsShared& S) {
  for (int r = 0; r <= P.K; ++r) {
    const uint32_t L = S.llen[r];
    if (L == KH_NOLIST || L == 0u) continue;
    uint32_t* gl = P.ws_lists + ((size_t)b * (P.K + 1) + r) * KH_KCAP;
    for (uint32_t e = threadIdx.x; e < L && e < (uint32_t)KH_KCAP; e += FT) gl[e] = 0u;
  }
}

// The sequence's rows are all done: acceptance in order from the drafted tokens'
// probabilities the row CTAs left, then the replacement or bonus token; writes
// the outputs (or hands the sequence to the cluster kernel) and re-arms the
// ticket, leaving the workspace zeroed.
__device__ __noinline__ void fs_finalize(const Params& P, int b, FsShared& S) {
  const int K = P.K, R2 = 2 * K + 1, tid = threadIdx.x;
  const KhRow* rr = P.ws_rowres + (size_t)b * R2;
  const float* tgt = static_cast<const float*>(P.rows0) + (size_t)b * (K + 1) * P.V;
  const float* drf = static_cast<const float*>(P.rows1) + (size_t)b * K * P.V;
  KF_MARK(b, 0);
  if (tid < 32) {
    uint32_t f = 0;
    for (int r = tid; r < R2; r += 32) f |= __ldcg(&rr[r].flags);
    if (tid <= K) S.llen[tid] = __ldcg(&rr[tid].pad[1]);
#pragma unroll
    for (int o = 16; o; o >>= 1) f |= __shfl_xor_sync(0xffffffffu, f, o);
    if (tid < K && !(f & (KH_ERR | KH_BAIL))) {
      const float p = __uint_as_float(__ldcg(&rr[tid].pad[0]));
      const float q = __uint_as_float(__ldcg(&rr[K + 1 + tid].pad[0]));
      uint32_t ku, kv;
      philox_uniform_bits(P.seed, philox_offset_of(P), (uint32_t)b, (uint32_t)tid, &ku, &kv);
      S.flag[tid] = __fmul_rn((float)ku * 5.9604644775390625e-08f, q) < p ? 1u : 0u;
    }
    if (tid == 0) S.flags = (int)f;
  }
  __syncthreads();
  const int flags = S.flags;
  if (tid == 0) {
    int n = K;
    if (!(flags & (KH_ERR | KH_BAIL)))
      for (int i = 0; i < K; ++i)
        if (!S.flag[i]) {
          n = i;
          break;
        }
    S.nacc = n;
  }
  __syncthreads();
  const int n = S.nacc;
  if (flags & KH_BAIL) {
    // the cluster kernel serves the sequence and clears the flag
    if (tid == 0) {
      P.ws_fb[b] = 1u;
      atomicOr(P.ws_work, 1u);
      P.ws_tickets[b] = 0u;
    }
    fs_clear_lists(P, b, S);
    __syncthreads();
    uint4* rz = reinterpret_cast<uint4*>(P.ws_rowres + (size_t)b * R2);
    for (int t = tid; t < 2 * R2; t += FT) rz[t] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  int tok = -1;
  if (!(flags & KH_ERR)) {
    const bool paired = n < K;
    const KhRow tp = kh_load_row(rr + n);
    const KhRow tq = paired ? kh_load_row(rr + K + 1 + n) : tp;
    uint32_t ku, kv;
    philox_uniform_bits(P.seed, philox_offset_of(P), (uint32_t)b, (uint32_t)n, &ku, &kv);
    const float* zp = tgt + (size_t)n * P.V;
    const float* zq = paired ? drf + (size_t)n * P.V : zp;
    const uint32_t L = tp.pad[1];
    KF_MARK(b, 1);
    KF_SET(b, 4, L != KH_NOLIST ? 1ull : 0ull);
    KF_SET(b, 5, (unsigned long long)n);
    if (L != KH_NOLIST) {
      tok = fs_sample_list(zp, zq, P.ws_lists + ((size_t)b * (K + 1) + n) * KH_KCAP, (int)L, paired,
                           kh_wof(tp), kh_wof(tq), kv, S);
    } else {
      tok = fs_sample_full(reinterpret_cast<const float4*>(zp), reinterpret_cast<const float4*>(zq), P.V / 4,
                           paired, kh_wof(tp), kh_wof(tq), kv, S);
    }
    KF_MARK(b, 2);
  }
  if (tid == 0) {
    const bool bad = (flags & KH_ERR) || tok < 0;
    int32_t* ot = P.out_tokens + (size_t)b * (K + 1);
    for (int q = 0; q <= K; ++q)
      ot[q] = bad ? -1 : (q < n ? P.dtok[(size_t)b * K + q] : (q == n ? tok : -1));
    P.out_n[b] = bad ? -1 : n;
    P.ws_tickets[b] = 0u;
  }
  fs_clear_lists(P, b, S);
  __syncthreads();
  uint4* rz = reinterpret_cast<uint4*>(P.ws_rowres + (size_t)b * R2);
  for (int t = tid; t < 2 * R2; t += FT) rz[t] = make_uint4(0u, 0u, 0u, 0u);
}

// Processing-order class of sequence b for fstream_kernel: 0 top-p without
// top-k (two or three passes per row and a full-row sample), 1 no truncation
// (one pass, full-row sample), 2 top-k (one pass, listed sample), 3 not served.
__device__ __forceinline__ int fs_seq_class(const Params& P, int b) {
  if (!fast_seq(P, b)) return 3;
  const int k = P.topk[b];
  if (k > 0 && k < P.V) return 2;
  return P.topp[b] < 1.0f ? 0 : 1;
}

// The batch's sequences in processing order, heaviest class first (so that the
// last rows handed out are short ones and the CTAs finish close together); the
// order within a class is immaterial (results depend on the sequence alone).
__global__ void __launch_bounds__(1024) fs_order_kernel(const Params P) {
  __shared__ uint32_t cnt[4], next[4];
  const int tid = threadIdx.x;
  if (tid < 4) cnt[tid] = 0u;
  __syncthreads();
  for (int b = tid; b < P.B; b += blockDim.x) atomicAdd(&cnt[fs_seq_class(P, b)], 1u);
  __syncthreads();
  if (tid == 0) {
    uint32_t a = 0u;
    for (int c = 0; c < 4; ++c) {
      next[c] = a;
      a += cnt[c];
    }
  }
  __syncthreads();
  for (int b = tid; b < P.B; b += blockDim.x) P.ws_perm[atomicAdd(&next[fs_seq_class(P, b)], 1u)] = b;
}

// Persistent CTAs take rows of the batch's sampled fp32 sequences from a work
// counter, sequence by sequence in the order fs_order_kernel set. Rows of other
// sequences are skipped.
__global__ void __launch_bounds__(FT, 2) fstream_kernel(const Params P, int nitems) {
  __shared__ FsShared S;
  // the cluster kernel may launch now; it waits for this grid before reading
  asm volatile("griddepcontrol.launch_dependents;");
  const int tid = threadIdx.x;
  const int K = P.K, R2 = 2 * K + 1;
  while (true) {
    if (tid == 0) S.item = (int)atomicAdd(P.ws_fnext, 1u);
    __syncthreads();
    const int item = S.item;
    __syncthreads();
    if (item >= nitems) break;
    const int pos_b = item / R2, r = item - pos_b * R2;
    const int b = P.ws_perm[pos_b];
    if (!fast_seq(P, b)) continue;
    const bool target = r <= K;
    const float* row = target ? static_cast<const float*>(P.rows0) + ((size_t)b * (K + 1) + r) * P.V
                              : static_cast<const float*>(P.rows1) + ((size_t)b * K + (r - K - 1)) * P.V;
    // the drafted token whose probability this row gives (target rows i < K, draft rows)
    const int pos = target ? r : r - K - 1;
    const int d = pos < K ? P.dtok[(size_t)b * K + pos] : -1;
    uint32_t* glist = target ? P.ws_lists + ((size_t)b * (K + 1) + r) * KH_KCAP : nullptr;
    KH_MARK(item, 0);
    const KhRow res = fs_row(row, P.V, P.temp[b], P.topk[b], P.topp[b], d, glist, S);
    KH_MARK(item, 4);
#ifdef SV_TRACE
    if (tid == 0 && item < 8192) {
      uint32_t smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      const int k = P.topk[b];
      const int cls = (k > 0 && k < P.V) ? FC_TOPK : (P.topp[b] < 1.0f ? FC_TOPP : FC_ALL);
      g_khtrace[item * 8 + 7] |= smid | ((unsigned long long)cls << 16) | ((unsigned long long)res.flags << 20);
    }
#endif
    if (tid == 0) {
      uint4* dst = reinterpret_cast<uint4*>(P.ws_rowres + (size_t)b * R2 + r);
      // a draft row never keeps a list: the sampling list is the target row's
      const uint32_t len = target ? res.pad[1] : KH_NOLIST;
      dst[0] = make_uint4(__float_as_uint(res.zt), __float_as_uint(res.invZ), __float_as_uint(res.m),
                          __float_as_uint(res.c));
      dst[1] = make_uint4((uint32_t)res.idcut, res.flags, res.pad[0], len);
      __threadfence();
      S.last = atomicAdd(&P.ws_tickets[b], 1u) == (unsigned int)(R2 - 1);
      if (S.last) __threadfence();
    }
    __syncthreads();
    if (S.last) {
      KH_MARK(item, 5);
      fs_finalize(P, b, S);
      KH_MARK(item, 6);
    }
    __syncthreads();
  }
  // finish only after greedy_kernel (launched before, possibly still running)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the last CTA to leave re-arms the work counter and clears the order
  if (tid == 0) {
    __threadfence();
    S.last = atomicAdd(P.ws_fdone, 1u) == gridDim.x - 1u;
  }
  __syncthreads();
  if (S.last) {
    for (int i = tid; i < P.B; i += FT) P.ws_perm[i] = 0;
    if (tid == 0) {
      *P.ws_fnext = 0u;
      *P.ws_fdone = 0u;
    }
  }
}

}  // namespace sv
