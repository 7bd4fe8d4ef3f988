// keyhist.cuh -- one-pass verify path for sampled sequences with bf16 rows.
//
// Included by spec_verify.cu (it uses Params, the Philox and fixed-point
// helpers and mass_threshold from there).
//
// One CTA owns one logit row at a time. It streams the row from HBM once and
// counts every 16-bit logit key into a shared-memory histogram whose bins are
// the distinct bf16 values (values with |z| < 2^-40 share one bin; their
// weights differ from 2^(-m*c) by less than 2^-24 relative for c < 2^16). The
// weight of a bin depends on its value alone, so a single sweep over the bins
// gives the exact fixed-point normaliser, the top-k count cut and the top-p
// mass cut: every cut falls on a bin, and a cut inside a bin of equal logits
// keeps the lowest token ids (a second, L2-resident read of the row finds the
// id). The row's result -- cut value, id cut, 1/Z, maximum, c -- goes to the
// workspace; the CTA that finishes the last of a sequence's 2K+1 rows runs the
// acceptance tests in order and draws the replacement from (p - q)+ or the
// bonus token from p_K with an inverse CDF in token-id order.
//
// Counts are packed two per 32-bit word (16 bits each). A bin holding more than
// 65535 equal logits carries into its neighbour; every such carry lowers the
// total count, so a total different from V hands the sequence to the cluster
// kernel, as does a cut inside the merged |z| < 2^-40 bin with a partial quota.
#pragma once

namespace sv {

constexpr int KT = 512;                                   // threads per CTA
constexpr int KWARP = KT / 32;
constexpr uint32_t KH_TSPLIT = 87u << 7;                  // |z| < 2^(87-127) = 2^-40
constexpr int KH_OFF = 0x7FFF - (int)KH_TSPLIT + 2;       // bin of the merged tiny values
constexpr int KH_TOP = 2 * KH_OFF - 1;                    // largest bin index (+NaN)
constexpr int KH_NW = KH_TOP / 2 + 1;                     // histogram words
constexpr int KH_WPT = (KH_NW + KT - 1) / KT;             // words swept per thread
constexpr int KH_NINF = KH_OFF - (0x7F80 - (int)KH_TSPLIT + 1);   // bin of -inf
constexpr int KH_PINF = KH_OFF + (0x7F80 - (int)KH_TSPLIT + 1);   // bin of +inf
constexpr int KH_PF = 4;                                  // 16-byte loads in flight per thread
constexpr int KH_MAXBLK = 64;                             // 32-vector blocks per warp range (V <= 262144)
constexpr size_t KH_HIST_BYTES = ((size_t)KH_NW * 4 + 15) & ~(size_t)15;
constexpr size_t KH_SMEM = KH_HIST_BYTES + 2 * (size_t)KWARP * KH_MAXBLK * 8;
constexpr float KH_LOG2E = 1.44269504088896341f;

constexpr uint32_t KH_ERR = 1u, KH_BAIL = 2u;
constexpr int KH_LCAP = 1024;                             // window candidates per target row
constexpr int KH_KCAP = 256;                              // kept-token list per target row (workspace)
constexpr uint32_t KH_NOLIST = 0xFFFFFFFFu;
constexpr float KH_LIST_BITS = 12.0f;                     // listed: weight >= 2^-12 of the maximum

#ifdef SV_TRACE
// Phase timestamps per row item (trace builds): 0 fetched, 1 streamed, 2 swept,
// 3 cut found, 4 row done, 5 finalize start, 6 finalize end, 7 SM id.
__device__ unsigned long long g_khtrace[8192 * 8];
#define KH_MARK(item, k)                                                   \
  do {                                                                     \
    if (threadIdx.x == 0 && (item) >= 0 && (item) < 8192) g_khtrace[(item) * 8 + (k)] = global_timer_ns(); \
  } while (0)
// Per-sequence finalize timestamps: 0 start, 1 acceptance done, 2 first sampling
// pass done, 3 end; 4 = redo, 5 = n.
__device__ unsigned long long g_kftrace[1024 * 8];
#define KF_MARK(b, k)                                                      \
  do {                                                                     \
    if (threadIdx.x == 0 && (b) >= 0 && (b) < 1024) g_kftrace[(b) * 8 + (k)] = global_timer_ns(); \
  } while (0)
#define KF_SET(b, k, v)                                                    \
  do {                                                                     \
    if (threadIdx.x == 0 && (b) >= 0 && (b) < 1024) g_kftrace[(b) * 8 + (k)] = (v);   \
  } while (0)
#else
#define KF_MARK(b, k) \
  do {                \
  } while (0)
#define KF_SET(b, k, v) \
  do {                  \
  } while (0)
#define KH_MARK(item, k) \
  do {                   \
  } while (0)
#endif

// Per-row result, written by the row's CTA and read by the sequence's finalizer.
struct KhRow {
  float zt;        // cut logit; kept iff z > zt or (z == zt and id <= idcut)
  float invZ;      // 2^44 / (fixed-point mass of the kept set)
  float m;         // row maximum
  float c;         // log2(e) / T
  int idcut;
  uint32_t flags;  // KH_ERR (NaN, +inf or no finite logit), KH_BAIL
  uint32_t pad[2];
};

// The row constants the sampling phase needs, passed by value (registers).
struct KhW {
  float zt, invZ, m, c;
  int idcut;
};
__device__ __forceinline__ KhW kh_wof(const KhRow& r) {
  KhW w;
  w.zt = r.zt;
  w.invZ = r.invZ;
  w.m = r.m;
  w.c = r.c;
  w.idcut = r.idcut;
  return w;
}

// Bin of a bf16 bit pattern; increasing in the logit's value.
__device__ __forceinline__ uint32_t kh_bin(uint32_t h) {
  const uint32_t t = max(h & 0x7FFFu, KH_TSPLIT - 1u) - (KH_TSPLIT - 1u);
  return (h & 0x8000u) ? (uint32_t)KH_OFF - t : (uint32_t)KH_OFF + t;
}
// The logit of a bin (0 for the merged tiny bin).
__device__ __forceinline__ float kh_value(int idx) {
  if (idx == KH_OFF) return 0.0f;
  const uint32_t t = (uint32_t)(idx > KH_OFF ? idx - KH_OFF : KH_OFF - idx);
  const uint32_t h = (t - 1u + KH_TSPLIT) | (idx < KH_OFF ? 0x8000u : 0u);
  return __uint_as_float(h << 16);
}
// Weight 2^((z - m) * c): the product is kept as an exact two-term sum and split
// into integer and fraction, so the fraction keeps full precision. 0 for -inf.
__device__ __forceinline__ float kh_w(float z, float m, float c) {
  const float d = z - m;
  const float hi = d * c;
  if (!(hi > -160.0f)) return 0.0f;
  const float lo = fmaf(d, c, -hi);
  const float n = rintf(hi);
  const float f = (hi - n) + lo;
  return ex2_approx(f) * pow2i((int)n);
}
__device__ __forceinline__ unsigned long long kh_fix(float z, float m, float c) {
  return fix_pow2(kh_w(z, m, c), FIX);
}
__device__ __forceinline__ bool kh_kept(float z, int id, float zt, int idcut) {
  return z > zt || (z == zt && id <= idcut);
}

// A sampled sequence served by this path: finite T > 0 with c < 2^16, valid
// top-k / top-p and drafted tokens in range (everything else, parameter errors
// included, goes to the cluster kernel).
__device__ __forceinline__ bool fast_seq(const Params& P, int b) {
  const float T = P.temp[b];
  if (!(T > 0.0f) || !(T < INFINITY) || !(P.topp[b] > 0.0f) || P.topk[b] < 0) return false;
  if (!(__fdiv_rn(KH_LOG2E, T) < 65536.0f)) return false;
  for (int q = 0; q < P.K; ++q) {
    const int d = P.dtok[(size_t)b * P.K + q];
    if (d < 0 || d >= P.V) return false;
  }
  return true;
}

struct KhShared {
  unsigned long long s64[KWARP];
  unsigned long long s64b[KWARP];
  uint32_t s32[KWARP];
  float fmax[KWARP];
  unsigned long long Mcut, Wcut;       // mass above the cut bin, its weight
  unsigned long long acc;              // sampling: exclusive sum before the crossing warp
  int cbin, cq, ccnt;                  // cut bin, quota, count
  int kbin, kq;
  unsigned long long Mk, Wk;
  int item, last, flags, idcut, wq, rq;
  int nacc, tok, useR;
  uint32_t need;                       // positions whose acceptance waits for a draft id split
  uint32_t llen[17];                   // kept-list lengths of the sequence's target rows
  uint32_t cmax;                       // collection: running block maximum (order-preserving key)
  uint32_t ccount;                     // collection: candidates pushed
  uint32_t gcount;                     // collection: kept tokens written out
  uint32_t flag[16];
  float pz[16], qz[16];                // p(d), and q(d) if d is kept
  uint32_t ku[16];
};

// Exclusive sums of a count and a mass in descending thread order (thread KT-1
// first), and their totals, in one pass.
__device__ __forceinline__ void kh_above2(uint32_t c, unsigned long long m, KhShared& S,
                                          uint32_t* cab, uint32_t* ctot,
                                          unsigned long long* mab, unsigned long long* mtot) {
  const int l = lane_id(), w = warp_id();
  uint32_t ic = c;
  unsigned long long im = m;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t tc = __shfl_down_sync(0xffffffffu, ic, o);
    const unsigned long long tm = __shfl_down_sync(0xffffffffu, im, o);
    if (l + o < 32) {
      ic += tc;
      im += tm;
    }
  }
  __syncthreads();
  if (l == 0) {
    S.s32[w] = ic;
    S.s64[w] = im;
  }
  __syncthreads();
  uint32_t oc = 0, tc = 0;
  unsigned long long om = 0, tm = 0;
#pragma unroll
  for (int i = 0; i < KWARP; ++i) {
    const uint32_t sc = S.s32[i];
    const unsigned long long sm = S.s64[i];
    if (i > w) {
      oc += sc;
      om += sm;
    }
    tc += sc;
    tm += sm;
  }
  *cab = oc + ic - c;
  *ctot = tc;
  *mab = om + im - m;
  *mtot = tm;
}

// Exclusive sums in descending thread order (thread KT-1 first) and the total.
template <typename T>
__device__ __forceinline__ T kh_above(T v, T* scratch, T* total) {
  const int l = lane_id(), w = warp_id();
  T incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T t = __shfl_down_sync(0xffffffffu, incl, o);
    if (l + o < 32) incl += t;
  }
  __syncthreads();
  if (l == 0) scratch[w] = incl;
  __syncthreads();
  T off = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < KWARP; ++i) {
    const T s = scratch[i];
    if (i > w) off += s;
    tot += s;
  }
  *total = tot;
  return off + incl - v;
}

__device__ __forceinline__ uint4 kh_ld(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 kh_ld_l2(const uint4* p) { return __ldcg(p); }

// Counts the 8 logits of one vector; returns their packed maximum.
__device__ __forceinline__ __nv_bfloat162 kh_count8(uint32_t* hist, const uint4& w) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t i0 = kh_bin(ws[k] & 0xFFFFu), i1 = kh_bin(ws[k] >> 16);
    atomicAdd(&hist[i0 >> 1], 1u << ((i0 & 1u) << 4));
    atomicAdd(&hist[i1 >> 1], 1u << ((i1 & 1u) << 4));
  }
  __nv_bfloat162 a, b, c, d;
  memcpy(&a, &w.x, 4);
  memcpy(&b, &w.y, 4);
  memcpy(&c, &w.z, 4);
  memcpy(&d, &w.w, 4);
  return __hmax2(__hmax2(a, b), __hmax2(c, d));
}

// Candidate list of a target row: every token within D of the running block
// maximum at the time it is read. The running maximum never exceeds the row
// maximum m, so the list holds every token with z >= m - D unless it overflowed
// (the count S.ccount then exceeds KH_LCAP and the list is not used). A vector's
// candidates take their slots with one atomic; once the list has overflowed no
// more are written.
__device__ __forceinline__ void kh_collect(const uint4& w, int v, __nv_bfloat162 vm2, float D,
                                           float* theta, KhShared& S, unsigned long long* list) {
  const float vm = fmaxf(__low2float(vm2), __high2float(vm2));
  if (!(vm >= *theta)) return;
  if (*reinterpret_cast<volatile uint32_t*>(&S.ccount) > (uint32_t)KH_LCAP) return;
  float smax = key_to_float(*reinterpret_cast<volatile uint32_t*>(&S.cmax));
  if (vm > smax) {
    atomicMax(&S.cmax, okey(vm));
    smax = vm;
  }
  *theta = smax - D;
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  uint32_t mk = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint32_t bits = (e & 1) ? ws[e >> 1] >> 16 : ws[e >> 1] & 0xFFFFu;
    mk |= (uint32_t)(__uint_as_float(bits << 16) >= *theta) << e;
  }
  if (!mk) return;
  uint32_t slot = atomicAdd(&S.ccount, (uint32_t)__popc(mk));
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (!((mk >> e) & 1u)) continue;
    const uint32_t bits = (e & 1) ? ws[e >> 1] >> 16 : ws[e >> 1] & 0xFFFFu;
    if (slot < (uint32_t)KH_LCAP) list[slot] = (unsigned long long)(v * 8 + e) | ((unsigned long long)bits << 32);
    ++slot;
  }
}

// Streams one row (nv 16-byte vectors) into the histogram; returns this
// thread's maximum (NaN is ignored here: NaN bins are checked afterwards).
// COLLECT: also lists the candidates of kh_collect (threshold seeded by the
// block maximum of the first load wave).
template <bool COLLECT>
__device__ __forceinline__ float kh_stream(const uint4* src, int nv, uint32_t* hist, float D,
                                           KhShared& S, unsigned long long* list) {
  const int tid = threadIdx.x;
  uint4 buf[KH_PF];
  const uint32_t NEG2 = 0xFF80FF80u;
#pragma unroll
  for (int p = 0; p < KH_PF; ++p) {
    const int q = tid + p * KT;
    buf[p] = q < nv ? kh_ld(src + q) : make_uint4(NEG2, NEG2, NEG2, NEG2);
  }
  __nv_bfloat162 m2 = __halves2bfloat162(__ushort_as_bfloat16((unsigned short)0xFF80u),
                                         __ushort_as_bfloat16((unsigned short)0xFF80u));
  float theta = -INFINITY;
  if (COLLECT) {
    __nv_bfloat162 f2 = m2;
#pragma unroll
    for (int p = 0; p < KH_PF; ++p) {
      __nv_bfloat162 a, b, c, d;
      memcpy(&a, &buf[p].x, 4);
      memcpy(&b, &buf[p].y, 4);
      memcpy(&c, &buf[p].z, 4);
      memcpy(&d, &buf[p].w, 4);
      f2 = __hmax2(f2, __hmax2(__hmax2(a, b), __hmax2(c, d)));
    }
    float fm = fmaxf(__low2float(f2), __high2float(f2));
#pragma unroll
    for (int o = 16; o; o >>= 1) fm = fmaxf(fm, __shfl_xor_sync(0xffffffffu, fm, o));
    if (tid == 0) {
      S.cmax = okey(-INFINITY);
      S.ccount = 0u;
      S.gcount = 0u;
    }
    __syncthreads();
    if (lane_id() == 0) atomicMax(&S.cmax, okey(fm));
    __syncthreads();
    theta = key_to_float(S.cmax) - D;
  }
  for (int q0 = tid; q0 < nv; q0 += KH_PF * KT) {
#pragma unroll
    for (int p = 0; p < KH_PF; ++p) {
      const int q = q0 + p * KT;
      if (q < nv) {
        const uint4 w = buf[p];
        const int qn = q + KH_PF * KT;
        if (qn < nv) buf[p] = kh_ld(src + qn);
        const __nv_bfloat162 vm2 = kh_count8(hist, w);
        m2 = __hmax2(m2, vm2);
        if (COLLECT) kh_collect(w, q, vm2, D, &theta, S, list);
      }
    }
  }
  return fmaxf(__low2float(m2), __high2float(m2));
}

// 8-bit mask (token-id order) of the logits in w whose bf16 pattern is hb.
__device__ __forceinline__ uint32_t kh_match8(const uint4& w, uint32_t hb) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  uint32_t mk = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    mk |= (uint32_t)((ws[k] & 0xFFFFu) == hb) << (2 * k);
    mk |= (uint32_t)((ws[k] >> 16) == hb) << (2 * k + 1);
  }
  return mk;
}

extern __shared__ __align__(16) uint32_t kh_dyn[];
// Per-(warp, block) partial results after the histogram: block j of warp w
// covers vectors [a0(w) + 32 j, a0(w) + 32 j + 32).
__device__ __forceinline__ unsigned long long* kh_blk0() {
  return reinterpret_cast<unsigned long long*>(reinterpret_cast<unsigned char*>(kh_dyn) + KH_HIST_BYTES);
}
__device__ __forceinline__ unsigned long long* kh_blk1() { return kh_blk0() + KWARP * KH_MAXBLK; }

// The id of the q-th (1-based) token, in id order, whose logit pattern is hb.
// Every warp counts matches per 32-vector block of its contiguous id range;
// warp 0 then locates the block holding the q-th match with two lane-parallel
// scans and finds the token in it. -1 if there are fewer than q matches.
__device__ __noinline__ int kh_tie(const uint4* src, int nv, uint32_t hb, int q, KhShared& S) {
  const int w = warp_id(), l = lane_id();
  const int cw = (nv + KWARP - 1) / KWARP;
  const int nb = (cw + 31) / 32;
  const int a0 = min(w * cw, nv), a1 = min(a0 + cw, nv);
  uint32_t* blk = reinterpret_cast<uint32_t*>(kh_blk0());
  uint32_t tot = 0;
  for (int j = 0; j < nb; j += 4) {
    uint4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = a0 + (j + u) * 32 + l;
      x[u] = (j + u < nb && v < a1) ? kh_ld_l2(src + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = a0 + (j + u) * 32 + l;
      const uint32_t c = warp_sum((uint32_t)__popc((j + u < nb && v < a1) ? kh_match8(x[u], hb) : 0u));
      if (l == 0 && j + u < nb) blk[w * KH_MAXBLK + j + u] = c;
      tot += c;
    }
  }
  if (l == 0) S.s32[w] = tot;
  __syncthreads();
  if (w == 0) {
    // the warp range, then the block, holding the q-th match
    const uint32_t own = l < KWARP ? S.s32[l] : 0u;
    uint32_t incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (l >= o) incl += t;
    }
    const uint32_t bw = __ballot_sync(0xffffffffu, l < KWARP && incl >= (uint32_t)q);
    int id = -1;
    if (bw) {
      const int ww = __ffs(bw) - 1;
      uint32_t r = (uint32_t)q - (__shfl_sync(0xffffffffu, incl, ww) - __shfl_sync(0xffffffffu, own, ww));
      const int wa0 = min(ww * cw, nv), wa1 = min(wa0 + cw, nv);
      // blocks of warp ww: lane l holds blocks 2l and 2l+1
      const uint32_t b0 = 2 * l < nb ? blk[ww * KH_MAXBLK + 2 * l] : 0u;
      const uint32_t b1 = 2 * l + 1 < nb ? blk[ww * KH_MAXBLK + 2 * l + 1] : 0u;
      uint32_t bi = b0 + b1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, bi, o);
        if (l >= o) bi += t;
      }
      const uint32_t bl = __ballot_sync(0xffffffffu, bi >= r);
      if (bl) {
        const int lb = __ffs(bl) - 1;
        const uint32_t before = __shfl_sync(0xffffffffu, bi - b0 - b1, lb);
        const uint32_t lb0 = __shfl_sync(0xffffffffu, b0, lb);
        int jb = 2 * lb;
        r -= before;
        if (r > lb0) {
          r -= lb0;
          ++jb;
        }
        // the block: one vector per lane, in id order
        const int v = wa0 + jb * 32 + l;
        const uint32_t mk = v < wa1 ? kh_match8(kh_ld_l2(src + v), hb) : 0u;
        const uint32_t cnt = __popc(mk);
        uint32_t ci = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t t = __shfl_up_sync(0xffffffffu, ci, o);
          if (l >= o) ci += t;
        }
        const uint32_t hit = __ballot_sync(0xffffffffu, ci >= r && ci - cnt < r);
        if (hit && l == __ffs(hit) - 1) {
          uint32_t need = r - (ci - cnt);
          for (int e = 0; e < 8; ++e)
            if ((mk >> e) & 1u)
              if (--need == 0u) {
                id = v * 8 + e;
                break;
              }
        }
        id = __reduce_max_sync(0xffffffffu, id);
      }
    }
    if (l == 0) S.idcut = id;
  }
  __syncthreads();
  return S.idcut;
}

// Weight of bin idx in fixed point (0 for -inf; NaN / +inf bins never get here).
__device__ __forceinline__ unsigned long long kh_binw(int idx, float m, float c) {
  return idx > KH_NINF ? kh_fix(kh_value(idx), m, c) : 0ull;
}

constexpr int KH_DEFER = -2;       // idcut of a partial cut bin not yet split by id

// Warp 0: walks the bins of thread range t (words [t*WPT, ...)) in descending
// order from the running count acc / mass M before the range, and stops at the
// first bin where the count reaches k (by_mass false) or the mass exceeds Y.
// Publishes the bin, its count and weight, and the count and mass before it.
__device__ __forceinline__ void kh_walk(const uint32_t* hist, int t, uint32_t acc,
                                        unsigned long long M, bool by_mass, uint32_t k,
                                        unsigned long long Y, float m, float c, KhShared& S) {
  const int l = lane_id();
  const int w0 = min(t * KH_WPT, KH_NW), w1 = min(w0 + KH_WPT, KH_NW);
  const int n = w1 - w0;
  for (int base = 0; base < n; base += 32) {
    const int pos = base + l;
    const int wd = w1 - 1 - pos;
    const uint32_t x = pos < n ? hist[wd] : 0u;
    const uint32_t chi = x >> 16, clo = x & 0xFFFFu;
    const unsigned long long Whi = chi ? kh_binw(2 * wd + 1, m, c) : 0ull;
    const unsigned long long Wlo = clo ? kh_binw(2 * wd, m, c) : 0ull;
    const uint32_t cw = chi + clo;
    const unsigned long long mw = chi * Whi + clo * Wlo;
    uint32_t ic = cw;
    unsigned long long im = mw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t tc = __shfl_up_sync(0xffffffffu, ic, o);
      const unsigned long long tm = __shfl_up_sync(0xffffffffu, im, o);
      if (l >= o) {
        ic += tc;
        im += tm;
      }
    }
    const bool cross = pos < n && (by_mass ? (M + im > Y) : (acc + ic >= k));
    const uint32_t bal = __ballot_sync(0xffffffffu, cross);
    if (bal) {
      if (l == __ffs(bal) - 1) {
        uint32_t a2 = acc + ic - cw;
        unsigned long long M2 = M + im - mw;
        const bool in_hi = chi != 0u && (by_mass ? (M2 + chi * Whi > Y) : (a2 + chi >= k));
        if (!in_hi) {
          a2 += chi;
          M2 += chi * Whi;
        }
        S.cbin = 2 * wd + (in_hi ? 1 : 0);
        S.ccnt = (int)(in_hi ? chi : clo);
        S.Wcut = in_hi ? Whi : Wlo;
        S.Mcut = M2;
        S.kq = (int)a2;                 // count before the bin
      }
      return;
    }
    acc += __shfl_sync(0xffffffffu, ic, 31);
    M += __shfl_sync(0xffffffffu, im, 31);
  }
}

// One row: histogram, maximum, normaliser, top-k / top-p cut and (target rows)
// the id split of a partial cut bin; a draft row's split is left to the
// sequence's finalizer, which needs it only for tokens on the cut value.
// Leaves the histogram zeroed. The result is returned in every thread.
__device__ __noinline__ KhRow kh_row(const __nv_bfloat16* row, int V, float T, int k, float topP,
                                     bool target, uint32_t* hist, KhShared& S, uint32_t* glist,
                                     int item) {
  const int tid = threadIdx.x, l = lane_id(), w = warp_id();
  const int nv = V / 8;
  const bool defer_tie = !target;
  const uint4* src = reinterpret_cast<const uint4*>(row);
  uint32_t* rcnt = reinterpret_cast<uint32_t*>(kh_blk0());      // per thread range
  unsigned long long* rmass =
      reinterpret_cast<unsigned long long*>(reinterpret_cast<unsigned char*>(kh_blk0()) + KT * 4);
  unsigned long long* clist = kh_blk1();                         // candidates (id | bits << 32)
  rcnt[tid] = 0u;
  rmass[tid] = 0ull;
  const float c = __fdiv_rn(KH_LOG2E, T);
  const float D = __fdiv_rn(KH_LIST_BITS, c);                    // z >= m - D: weight >= 2^-12
  float mt = target ? kh_stream<true>(src, nv, hist, D, S, clist)
                    : kh_stream<false>(src, nv, hist, D, S, clist);
#pragma unroll
  for (int o = 16; o; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
  if (l == 0) S.fmax[w] = mt;
  __syncthreads();                              // the histogram is complete
  KH_MARK(item, 1);
  float m = S.fmax[0];
#pragma unroll
  for (int i = 1; i < KWARP; ++i) m = fmaxf(m, S.fmax[i]);

  // sweep, words interleaved over the threads (occupied bins cluster in a few
  // value ranges): counts and fixed-point masses, added to the word's thread range
  uint32_t bad = 0;
  // a lane's words are summed locally and added to their thread range once
  int rcur = -1;
  uint32_t cacc = 0;
  unsigned long long macc = 0;
  auto flush = [&]() {
    if (rcur >= 0 && cacc) {
      atomicAdd(&rcnt[rcur], cacc);
      if (macc) atomicAdd(&rmass[rcur], macc);
    }
    cacc = 0;
    macc = 0;
  };
  auto sweep_word = [&](int wd, uint32_t x) {
    const uint32_t chi = x >> 16, clo = x & 0xFFFFu;
    const int i0 = 2 * wd;
    if ((clo && (i0 < KH_NINF || i0 >= KH_PINF)) || (chi && (i0 + 1 < KH_NINF || i0 + 1 >= KH_PINF)))
      bad = 1u;
    const unsigned long long mw = (clo ? clo * kh_binw(i0, m, c) : 0ull) +
                                  (chi ? chi * kh_binw(i0 + 1, m, c) : 0ull);
    const int r = wd / KH_WPT;
    if (r != rcur) {
      flush();
      rcur = r;
    }
    cacc += chi + clo;
    macc += mw;
  };
  // four words per 16-byte load; the last word (an odd count) separately
  const uint4* h4 = reinterpret_cast<const uint4*>(hist);
  for (int v4 = tid; v4 < KH_NW / 4; v4 += KT) {
    const uint4 x = h4[v4];
    if ((x.x | x.y | x.z | x.w) == 0u) continue;
    if (x.x) sweep_word(4 * v4, x.x);
    if (x.y) sweep_word(4 * v4 + 1, x.y);
    if (x.z) sweep_word(4 * v4 + 2, x.z);
    if (x.w) sweep_word(4 * v4 + 3, x.w);
    flush();
  }
  for (int wd = (KH_NW / 4) * 4 + tid; wd < KH_NW; wd += KT)
    if (hist[wd]) sweep_word(wd, hist[wd]);
  flush();
  const int anyb = __syncthreads_or((int)bad);
  const uint32_t cnt = rcnt[tid];
  const unsigned long long mass = anyb ? 0ull : rmass[tid];
  uint32_t ctot, cab;
  unsigned long long Ztot, mab;
  kh_above2(cnt, mass, S, &cab, &ctot, &mab, &Ztot);
  KH_MARK(item, 2);

  KhRow res;
  res.m = m;
  res.c = c;
  res.zt = -INFINITY;
  res.idcut = V;
  res.invZ = 0.0f;
  res.flags = 0u;
  res.pad[0] = 0u;
  res.pad[1] = KH_NOLIST;
  if (anyb || !(m > -INFINITY)) res.flags = KH_ERR;
  else if (ctot != (uint32_t)V) res.flags = KH_BAIL;
  const bool topk = k > 0 && k < V;
  const bool topp = topP < 1.0f;
  unsigned long long ZL1 = Ztot;
  if (res.flags == 0u && topk) {
    // the bin holding the k-th token in (logit desc, id asc) order
    if (cab < (uint32_t)k && (uint32_t)k <= cab + cnt) {
      S.wq = tid;
      S.acc = mab;
      S.rq = (int)cab;
    }
    __syncthreads();
    if (w == 0) kh_walk(hist, S.wq, (uint32_t)S.rq, S.acc, false, (uint32_t)k, 0ull, m, c, S);
    __syncthreads();
    ZL1 = S.Mcut + (unsigned long long)(k - S.kq) * S.Wcut;
    if (!topp && tid == 0) S.cq = k - S.kq;   // tokens of the bin inside the top k
  }
  if (res.flags == 0u && topp) {
    // the bin where the exclusive mass first exceeds Y = the largest integer
    // below P * Z(L1); tokens with exclusive mass <= Y are kept
    const unsigned long long Y = mass_threshold(topP, ZL1);
    __syncthreads();
    if (mab <= Y && Y < mab + mass) {
      S.wq = tid;
      S.acc = mab;
      S.rq = (int)cab;
    }
    __syncthreads();
    if (w == 0) {
      kh_walk(hist, S.wq, (uint32_t)S.rq, S.acc, true, 0u, Y, m, c, S);
      __syncwarp();
      if (l == 0) S.cq = (int)((Y - S.Mcut) / S.Wcut) + 1;
    }
    __syncthreads();
  }
  // the histogram is not read again for this row
  for (int wd = tid; wd < KH_NW; wd += KT) hist[wd] = 0u;
  KH_MARK(item, 3);
  if (res.flags != 0u) return res;

  unsigned long long Zk = Ztot;
  // a target row's candidate list holds every kept token when the cut lies
  // within D of the maximum and the list did not overflow
  const uint32_t ncand = target ? S.ccount : 0u;
  bool listed = false;
  if (topk || topp) {
    const int cbin = S.cbin, q = S.cq, ccnt = S.ccnt;
    Zk = S.Mcut + (unsigned long long)q * S.Wcut;
    // kept tokens: those before the cut bin plus the bin's quota
    const int nkept = S.kq + min(q, ccnt);
    listed = target && ncand <= (uint32_t)KH_LCAP && cbin != KH_OFF && kh_value(cbin) >= m - D &&
             nkept <= KH_KCAP;
    if (q >= ccnt || S.Wcut == 0ull) {
      // the whole bin is kept (zero-weight tokens have p = 0 either way)
      if (cbin == KH_OFF) {
        res.zt = -__uint_as_float(KH_TSPLIT << 16);   // the value just below the bin
        res.idcut = -1;
      } else {
        res.zt = kh_value(cbin);
        res.idcut = V;
      }
    } else if (cbin == KH_OFF) {
      res.flags = KH_BAIL;                            // unequal logits share the bin
      return res;
    } else {
      res.zt = kh_value(cbin);
      res.pad[0] = (uint32_t)q;
      const uint32_t hb = __float_as_uint(res.zt) >> 16;
      if (defer_tie) {
        res.idcut = KH_DEFER;
      } else if (listed) {
        // the q-th lowest id among the listed tokens on the cut value
        if (tid == 0) S.idcut = -1;
        __syncthreads();
        for (uint32_t e = tid; e < ncand; e += KT) {
          const unsigned long long x = clist[e];
          if ((uint32_t)(x >> 32) != hb) continue;
          const uint32_t id = (uint32_t)x;
          int rank = 0;
          for (uint32_t f = 0; f < ncand; ++f) {
            const unsigned long long y = clist[f];
            rank += ((uint32_t)(y >> 32) == hb && (uint32_t)y < id) ? 1 : 0;
          }
          if (rank == q - 1) S.idcut = (int)id;
        }
        __syncthreads();
        res.idcut = S.idcut;
        if (res.idcut < 0) res.flags = KH_BAIL;
      } else {
        res.idcut = kh_tie(src, nv, hb, q, S);
        if (res.idcut < 0) res.flags = KH_BAIL;
      }
    }
  }
  if (listed && res.flags == 0u) {
    // the kept tokens, in no particular order
    for (uint32_t e = tid; e < ncand; e += KT) {
      const unsigned long long x = clist[e];
      const int id = (int)(uint32_t)x;
      if (kh_kept(__uint_as_float((uint32_t)(x >> 32) << 16), id, res.zt, res.idcut))
        glist[atomicAdd(&S.gcount, 1u)] = (uint32_t)id;
    }
    __syncthreads();
    res.pad[1] = S.gcount;
  }
  res.invZ = __fdiv_rn(17592186044416.0f, (float)Zk);   // 2^44 / Z
  return res;
}

// Sampling weights of one token: r = (p - q)+ and p, both 0 outside the
// target's kept set (probabilities in fp32, as 2^44-frame weights times 1/Z).
__device__ __forceinline__ void kh_elem(float zp, float zq, int id, bool paired, KhW tp, KhW tq,
                                        float* r, float* p) {
  *r = 0.0f;
  *p = 0.0f;
  if (kh_kept(zp, id, tp.zt, tp.idcut)) {
    const float pp = __fmul_rn(kh_w(zp, tp.m, tp.c), tp.invZ);
    float q = 0.0f;
    if (paired && kh_kept(zq, id, tq.zt, tq.idcut)) q = __fmul_rn(kh_w(zq, tq.m, tq.c), tq.invZ);
    *r = fmaxf(__fsub_rn(pp, q), 0.0f);
    *p = pp;
  }
}
__device__ __forceinline__ float kh_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float kh_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// Fixed-point (2^-40) residual and target masses of the 8 tokens of vector v
// (target logits a already loaded), for a vector holding a token of the
// target's kept set. *dhit is set when such a token sits on the draft row's
// cut value while that cut's id split is still deferred (its q is then not
// known yet).
#ifdef SV_TRACE
__device__ unsigned long long g_khheavy;
#endif
__device__ __noinline__ void kh_vec_heavy(uint4 a, const uint4* sq, int v, bool paired, KhW tp,
                                          KhW tq, unsigned long long* R, unsigned long long* Pm,
                                          bool* dhit) {
#ifdef SV_TRACE
  atomicAdd(&g_khheavy, 1ull);
#endif
  uint4 bq = make_uint4(0u, 0u, 0u, 0u);
  if (paired) bq = kh_ld_l2(sq + v);
  const uint32_t as[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bs[4] = {bq.x, bq.y, bq.z, bq.w};
  unsigned long long ra = 0, pa = 0;
  bool hit = false;
#pragma unroll 1
  for (int e = 0; e < 8; ++e) {
    const uint32_t xa = as[e >> 1], xb = bs[e >> 1];
    const float zp = (e & 1) ? kh_hi(xa) : kh_lo(xa);
    const float zq = (e & 1) ? kh_hi(xb) : kh_lo(xb);
    const int id = v * 8 + e;
    float r, p;
    kh_elem(zp, zq, id, paired, tp, tq, &r, &p);
    ra += fixr(r);
    pa += fixr(p);
    hit |= paired && tq.idcut == KH_DEFER && zq == tq.zt && kh_kept(zp, id, tp.zt, tp.idcut);
  }
  *R = ra;
  *Pm = pa;
  if (hit) *dhit = true;
}
// Whether vector a holds a logit >= zt (packed bf16 compares): a necessary
// condition for a kept token; zt2 holds the cut value (a bf16 value) twice.
__device__ __forceinline__ bool kh_vec_cand(const uint4& a, __nv_bfloat162 zt2) {
  __nv_bfloat162 x0, x1, x2, x3;
  memcpy(&x0, &a.x, 4);
  memcpy(&x1, &a.y, 4);
  memcpy(&x2, &a.z, 4);
  memcpy(&x3, &a.w, 4);
  return (__hge2_mask(x0, zt2) | __hge2_mask(x1, zt2) | __hge2_mask(x2, zt2) | __hge2_mask(x3, zt2)) != 0u;
}

// Warp sum of per-lane fixed-point masses below 2^51 (a vector's 8 weights of at
// most 16 * 2^40 each), as two 32-bit lane reductions of the low 24 bits and the
// rest: neither partial sum can overflow 32 bits.
__device__ __forceinline__ unsigned long long kh_wsum(unsigned long long x) {
  const uint32_t lo = __reduce_add_sync(0xffffffffu, (uint32_t)x & 0xFFFFFFu);
  const uint32_t hi = __reduce_add_sync(0xffffffffu, (uint32_t)(x >> 24));
  return ((unsigned long long)hi << 24) + lo;
}
// Weight tables of the sampling pass. A table holds one entry per bin from the
// cut bin to the bin of the row maximum, except the bins of 2^-40 <= |z| < 2^-8
// and the merged bin (a band around zero), whose rare tokens are evaluated
// directly: without the band a table across zero would need ~10k entries.
constexpr int KH_BAND = 32 * 128;
// Table slot of a bin outside the band, -1 inside it; increasing in the bin.
__device__ __forceinline__ int kh_slot(int bin) {
  return bin > KH_OFF + KH_BAND ? bin - (2 * KH_BAND + 1) : (bin < KH_OFF - KH_BAND ? bin : -1);
}
__device__ __forceinline__ int kh_slot_bin(int s) {
  return s >= KH_OFF - KH_BAND ? s + (2 * KH_BAND + 1) : s;
}
// Slots [*lo, *lo + *n) of the bins a cut at zt can keep on a row with maximum m.
__device__ __forceinline__ void kh_slots(float zt, float m, int* lo, int* n) {
  const int bz = zt > -INFINITY ? (int)kh_bin(__float_as_uint(zt) >> 16) : KH_NINF + 1;
  const int bm = (int)kh_bin(__float_as_uint(m) >> 16);
  const int l = bz < KH_OFF - KH_BAND ? bz : (bz > KH_OFF + KH_BAND ? bz - (2 * KH_BAND + 1) : KH_OFF - KH_BAND);
  const int h = bm < KH_OFF - KH_BAND ? bm : (bm > KH_OFF + KH_BAND ? bm - (2 * KH_BAND + 1) : KH_OFF - KH_BAND - 1);
  *lo = l;
  *n = h - l + 1;
}
// p of one token from a float table (or directly, in the band).
__device__ __forceinline__ float kh_ptab(uint32_t h, float z, const KhW& w, const float* tab, int lo,
                                         int n) {
  const int sl = kh_slot((int)kh_bin(h)) - lo;
  if ((unsigned)sl < (unsigned)n) return tab[sl];
  return __fmul_rn(kh_w(z, w.m, w.c), w.invZ);
}
// kh_vec_heavy with table lookups. Unpaired: tab64 holds fixr(p) per slot (w0 is
// the weight of z = 0). Paired: tab holds p per slot, then q per slot at tab + np.
// The weights are the ones kh_elem computes, so the sums match bit for bit.
__device__ __forceinline__ void kh_vec_tab(uint4 a, const uint4* sq, int v, bool paired,
                                           const KhW& tp, const KhW& tq, const float* tab,
                                           const unsigned long long* tab64, unsigned long long w0,
                                           int lop, int np, int loq, int nq, int cp, int cn,
                                           int idcut0, unsigned long long* R,
                                           unsigned long long* Pm, bool* dhit) {
  uint4 bq = make_uint4(0u, 0u, 0u, 0u);
  if (paired) bq = kh_ld_l2(sq + v);
  const uint32_t as[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bs[4] = {bq.x, bq.y, bq.z, bq.w};
  unsigned long long ra = 0, pa = 0;
  bool hit = false;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint32_t hp = (e & 1) ? as[e >> 1] >> 16 : as[e >> 1] & 0xFFFFu;
    const float zp = __uint_as_float(hp << 16);
    const int id = v * 8 + e;
    if (!paired) {
      // table index straight from the bits (slot - lo: a + cp above zero, cn - a
      // below); below the cut it is negative, and the cut bin itself is index 0
      // when the cut lies outside the band (idcut0 = its id cut, else INT_MAX)
      const int a16 = (int)(hp & 0x7FFFu);
      if (a16 < (int)KH_TSPLIT + KH_BAND) {
        if (kh_kept(zp, id, tp.zt, tp.idcut))
          pa += a16 == 0 ? w0 : fixr(__fmul_rn(kh_w(zp, tp.m, tp.c), tp.invZ));
        continue;
      }
      const int ix = (hp & 0x8000u) ? cn - a16 : a16 + cp;
      const bool in = (unsigned)ix < (unsigned)np && (ix != 0 || id <= idcut0);
      pa += in ? tab64[ix] : 0ull;
      continue;
    }
    if (!kh_kept(zp, id, tp.zt, tp.idcut)) continue;
    const float pp = kh_ptab(hp, zp, tp, tab, lop, np);
    const uint32_t hq = (e & 1) ? bs[e >> 1] >> 16 : bs[e >> 1] & 0xFFFFu;
    const float zq = __uint_as_float(hq << 16);
    const float q = kh_kept(zq, id, tq.zt, tq.idcut) ? kh_ptab(hq, zq, tq, tab + np, loq, nq) : 0.0f;
    hit |= tq.idcut == KH_DEFER && zq == tq.zt;
    ra += fixr(fmaxf(__fsub_rn(pp, q), 0.0f));
    pa += fixr(pp);
  }
  *R = paired ? ra : pa;
  *Pm = pa;
  if (hit) *dhit = true;
}

// Inverse CDF in token-id order over (p - q)+ (paired) or p: the smallest id j
// whose running sum S_j satisfies S_j * 2^24 > kv * S (S the total); when the
// residual mass is 0 the target p is used. Every warp sums its contiguous id
// range per 32-vector block; warp 0 locates the crossing block with two
// lane-parallel scans and walks it. -1 if no token qualifies.
__device__ __noinline__ int kh_sample(const uint4* sp, const uint4* sq, int nv, bool paired,
                                      const KhW tp, const KhW tq, uint32_t kv, KhShared& S, int bt) {
  const int w = warp_id(), l = lane_id();
  const int cw = (nv + KWARP - 1) / KWARP;
  const int nb = (cw + 31) / 32;
  const int a0 = min(w * cw, nv), a1 = min(a0 + cw, nv);
  unsigned long long* bR = kh_blk0();
  unsigned long long* bP = kh_blk1();
  unsigned long long tR = 0, tP = 0;
  bool dhit = false;
  const __nv_bfloat162 zt2 = __float2bfloat162_rn(tp.zt);   // zt is a bf16 value
  // When the bins a cut keeps fit the histogram's shared memory (zero here), the
  // weights are tabulated per bin once and the pass reads them instead of
  // evaluating exp2 per token; the table is zeroed again afterwards.
  float* tab = reinterpret_cast<float*>(kh_dyn);
  unsigned long long* tab64 = reinterpret_cast<unsigned long long*>(kh_dyn);
  int lop, np, loq = 0, nq = 0;
  kh_slots(tp.zt, tp.m, &lop, &np);
  if (paired) kh_slots(tq.zt, tq.m, &loq, &nq);
  np = max(np, 0);
  nq = max(nq, 0);
  const int twords = paired ? np + nq : 2 * np;  // 32-bit words the table takes
  const bool use_tab = twords <= KH_NW;
  const unsigned long long w0 = fixr(__fmul_rn(kh_w(0.0f, tp.m, tp.c), tp.invZ));
  // unpaired index constants: a bf16 magnitude a outside the band has slot
  // a + (KH_OFF - KH_TSPLIT - 2 KH_BAND) when positive, KH_OFF + KH_TSPLIT - 1 - a when negative
  const int cp = KH_OFF - (int)KH_TSPLIT - 2 * KH_BAND - lop;
  const int cn = KH_OFF + (int)KH_TSPLIT - 1 - lop;
  const int idcut0 =
      (int)(__float_as_uint(tp.zt) >> 16 & 0x7FFFu) >= (int)KH_TSPLIT + KH_BAND && tp.zt > -INFINITY
          ? tp.idcut : INT_MAX;
  if (use_tab) {
    for (int j = threadIdx.x; j < np + nq; j += KT) {
      const bool isq = j >= np;
      const KhW& w = isq ? tq : tp;
      const float z = kh_value(kh_slot_bin(isq ? loq + (j - np) : lop + j));
      const float pz = __fmul_rn(kh_w(z, w.m, w.c), w.invZ);
      if (paired) tab[j] = pz;
      else tab64[j] = fixr(pz);
    }
    __syncthreads();
  }
  constexpr int U = 4;                          // target vectors in flight per lane
  for (int j = 0; j < nb; j += U) {
    uint4 av[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = a0 + (j + u) * 32 + l;
      av[u] = (j + u < nb && v < a1) ? kh_ld_l2(sp + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (j + u < nb) {
        const int v = a0 + (j + u) * 32 + l;
        const bool cand = v < a1 && kh_vec_cand(av[u], zt2);
        unsigned long long r = 0, p = 0;
        // blocks without a kept target token contribute nothing
        if (__any_sync(0xffffffffu, cand)) {
          if (cand) {
            if (use_tab)
              kh_vec_tab(av[u], sq, v, paired, tp, tq, tab, tab64, w0, lop, np, loq, nq, cp, cn, idcut0,
                         &r, &p, &dhit);
            else kh_vec_heavy(av[u], sq, v, paired, tp, tq, &r, &p, &dhit);
          }
          p = kh_wsum(p);
          r = paired ? kh_wsum(r) : p;
        }
        if (l == 0) {
          bR[w * KH_MAXBLK + j + u] = r;
          bP[w * KH_MAXBLK + j + u] = p;
        }
        tR += r;
        tP += p;
      }
    }
  }
  if (l == 0) {
    S.s64[w] = tR;
    S.s64b[w] = tP;
  }
  const bool redo = __syncthreads_or(dhit ? 1 : 0) != 0;
  if (use_tab) {
    for (int j = threadIdx.x; j < twords; j += KT) tab[j] = 0.0f;
    __syncthreads();
  }
  if (redo) return -2;                          // the caller splits the draft cut first
  KF_MARK(bt, 6);
  if (w == 0) {
    const unsigned long long oR = l < KWARP ? S.s64[l] : 0ull, oP = l < KWARP ? S.s64b[l] : 0ull;
    const unsigned long long SR = warp_sum(oR), SP = warp_sum(oP);
    const bool useR = SR > 0ull;
    const unsigned long long St = useR ? SR : SP;
    const unsigned long long* bv = useR ? bR : bP;
    const unsigned long long own = useR ? oR : oP;
    unsigned long long incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
      if (l >= o) incl += t;
    }
    const uint32_t bw = __ballot_sync(0xffffffffu, l < KWARP && mul_gt(incl, 1ull << 24, kv, St));
    int tok = -1;
    if (bw) {
      const int ww = __ffs(bw) - 1;
      unsigned long long acc = __shfl_sync(0xffffffffu, incl - own, ww);
      const int wa0 = min(ww * cw, nv), wa1 = min(wa0 + cw, nv);
      const unsigned long long b0 = 2 * l < nb ? bv[ww * KH_MAXBLK + 2 * l] : 0ull;
      const unsigned long long b1 = 2 * l + 1 < nb ? bv[ww * KH_MAXBLK + 2 * l + 1] : 0ull;
      unsigned long long bi = b0 + b1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, bi, o);
        if (l >= o) bi += t;
      }
      const uint32_t bl = __ballot_sync(0xffffffffu, mul_gt(acc + bi, 1ull << 24, kv, St));
      if (bl) {
        const int lb = __ffs(bl) - 1;
        acc += __shfl_sync(0xffffffffu, bi - b0 - b1, lb);
        const unsigned long long lb0 = __shfl_sync(0xffffffffu, b0, lb);
        int jb = 2 * lb;
        if (!mul_gt(acc + lb0, 1ull << 24, kv, St)) {
          acc += lb0;
          ++jb;
        }
        // the block: one vector per lane, in id order
        const int v = wa0 + jb * 32 + l;
        unsigned long long r = 0, p = 0;
        bool dh = false;
        if (v < wa1) {
          const uint4 a = kh_ld_l2(sp + v);
          if (kh_vec_cand(a, zt2)) kh_vec_heavy(a, sq, v, paired, tp, tq, &r, &p, &dh);
        }
        const unsigned long long mine = useR ? r : p;
        unsigned long long ci = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned long long t = __shfl_up_sync(0xffffffffu, ci, o);
          if (l >= o) ci += t;
        }
        const uint32_t hit = __ballot_sync(0xffffffffu, v < wa1 && mul_gt(acc + ci, 1ull << 24, kv, St));
        if (hit && l == __ffs(hit) - 1) {
          // walk this vector's tokens in id order
          const uint4 a = kh_ld_l2(sp + v);
          uint4 b = make_uint4(0u, 0u, 0u, 0u);
          if (paired) b = kh_ld_l2(sq + v);
          const uint32_t as[4] = {a.x, a.y, a.z, a.w}, bs[4] = {b.x, b.y, b.z, b.w};
          unsigned long long run = acc + ci - mine;
          for (int e = 0; e < 8 && tok < 0; ++e) {
            const uint32_t xa = as[e >> 1], xb = bs[e >> 1];
            const float zp = (e & 1) ? kh_hi(xa) : kh_lo(xa);
            const float zq = (e & 1) ? kh_hi(xb) : kh_lo(xb);
            float rr, pp;
            kh_elem(zp, zq, v * 8 + e, paired, tp, tq, &rr, &pp);
            run += fixr(useR ? rr : pp);
            if (mul_gt(run, 1ull << 24, kv, St)) tok = v * 8 + e;
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

// Exclusive sums in ascending thread order and the total.
template <typename T>
__device__ __forceinline__ T kh_below(T v, T* scratch, T* total) {
  const int l = lane_id(), w = warp_id();
  T incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T t = __shfl_up_sync(0xffffffffu, incl, o);
    if (l >= o) incl += t;
  }
  __syncthreads();
  if (l == 31) scratch[w] = incl;
  __syncthreads();
  T off = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < KWARP; ++i) {
    const T s = scratch[i];
    if (i < w) off += s;
    tot += s;
  }
  *total = tot;
  return off + incl - v;
}

// The inverse CDF of kh_sample over a target row whose kept tokens are listed
// (L <= KH_LCAP ids, any order): only listed tokens carry p > 0, so the sums run
// over the list sorted by id. Uses the histogram's shared memory as scratch and
// zeroes it again. -2 when a listed token sits on the draft row's deferred cut
// value (the caller splits that cut first), -1 if no token qualifies.
__device__ __noinline__ int kh_sample_list(const unsigned short* zp_row, const unsigned short* zq_row,
                                           const uint32_t* glist, int L, bool paired, KhW tp, KhW tq,
                                           uint32_t kv, KhShared& S) {
  const int tid = threadIdx.x;
  uint32_t* ids = kh_dyn;                                          // [KH_LCAP]
  unsigned long long* wr = reinterpret_cast<unsigned long long*>(kh_dyn + KH_LCAP);   // [KH_LCAP] r, sorted
  unsigned long long* wp = wr + KH_LCAP;                           // [KH_LCAP] p, sorted
  uint32_t* sid = reinterpret_cast<uint32_t*>(wp + KH_LCAP);       // [KH_LCAP] ids, sorted
  bool dhit = false;
  for (int e = tid; e < L; e += KT) ids[e] = __isShared(glist) ? glist[e] : __ldcg(glist + e);
  __syncthreads();
  for (int e = tid; e < L; e += KT) {
    const int id = (int)ids[e];
    const float zp = __uint_as_float((uint32_t)__ldcg(zp_row + id) << 16);
    const float zq = paired ? __uint_as_float((uint32_t)__ldcg(zq_row + id) << 16) : 0.0f;
    float r, p;
    kh_elem(zp, zq, id, paired, tp, tq, &r, &p);
    dhit |= paired && tq.idcut == KH_DEFER && zq == tq.zt;
    int rank = 0;
    for (int f = 0; f < L; ++f) rank += (int)(ids[f] < (uint32_t)id);
    wr[rank] = fixr(r);
    wp[rank] = fixr(p);
    sid[rank] = (uint32_t)id;
  }
  const bool redo = __syncthreads_or(dhit ? 1 : 0) != 0;
  int tok = -2;
  if (!redo) {
    // two consecutive sorted entries per thread
    const int e0 = 2 * tid;
    unsigned long long r2 = 0, p2 = 0;
    if (e0 < L) {
      r2 += wr[e0];
      p2 += wp[e0];
    }
    if (e0 + 1 < L) {
      r2 += wr[e0 + 1];
      p2 += wp[e0 + 1];
    }
    unsigned long long SR, SP;
    const unsigned long long xr = kh_below<unsigned long long>(r2, S.s64, &SR);
    const unsigned long long xp = kh_below<unsigned long long>(p2, S.s64b, &SP);
    const bool useR = SR > 0ull;
    const unsigned long long St = useR ? SR : SP;
    if (tid == 0) S.tok = -1;
    __syncthreads();
    unsigned long long run = useR ? xr : xp;
    for (int e = e0; e < min(e0 + 2, L); ++e) {
      const unsigned long long own = useR ? wr[e] : wp[e];
      if (!mul_gt(run, 1ull << 24, kv, St) && mul_gt(run + own, 1ull << 24, kv, St)) S.tok = (int)sid[e];
      run += own;
    }
    __syncthreads();
    tok = S.tok;
  }
  // restore the histogram's zeros
  uint4* z4 = reinterpret_cast<uint4*>(kh_dyn);
  const int n16 = (KH_LCAP * 4 + 2 * KH_LCAP * 8 + KH_LCAP * 4) / 16;
  for (int t = tid; t < n16; t += KT) z4[t] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  return tok;
}

__device__ __forceinline__ float kh_ldz(const void* rows, size_t row, int V, int id) {
  const unsigned short h =
      __ldg(reinterpret_cast<const unsigned short*>(rows) + row * (size_t)V + (size_t)id);
  return __uint_as_float((uint32_t)h << 16);
}
__device__ __forceinline__ KhRow kh_load_row(const KhRow* p) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  const uint4 a = __ldcg(q), b = __ldcg(q + 1);
  KhRow r;
  r.zt = __uint_as_float(a.x);
  r.invZ = __uint_as_float(a.y);
  r.m = __uint_as_float(a.z);
  r.c = __uint_as_float(a.w);
  r.idcut = (int)b.x;
  r.flags = b.y;
  r.pad[0] = b.z;
  r.pad[1] = b.w;
  return r;
}

// Number of tokens with id < id_end whose logit pattern is hb (CTA-wide).
__device__ __noinline__ uint32_t kh_rank_before(const uint4* src, int id_end, uint32_t hb, KhShared& S) {
  const int nfull = id_end / 8, rem = id_end % 8;
  uint32_t n = 0;
  for (int v = threadIdx.x; v < nfull; v += KT) n += __popc(kh_match8(kh_ld_l2(src + v), hb));
  if (threadIdx.x == 0 && rem) n += __popc(kh_match8(kh_ld_l2(src + nfull), hb) & ((1u << rem) - 1u));
  n = warp_sum(n);
  __syncthreads();
  if (lane_id() == 0) S.s32[warp_id()] = n;
  __syncthreads();
  uint32_t t = 0;
#pragma unroll
  for (int i = 0; i < KWARP; ++i) t += S.s32[i];
  __syncthreads();
  return t;
}

// Clears the kept-token lists of sequence b's target rows (the call leaves the
// workspace zeroed); their lengths were read from the row results into S.llen.
__device__ __noinline__ void kh_clear_lists(const Params& P, int b, const KhShared& S) {
  for (int r = 0; r <= P.K; ++r) {
    const uint32_t L = S.llen[r];
    if (L == KH_NOLIST || L == 0u) continue;
    uint32_t* gl = P.ws_lists + ((size_t)b * (P.K + 1) + r) * KH_KCAP;
    for (uint32_t e = threadIdx.x; e < L && e < (uint32_t)KH_KCAP; e += KT) gl[e] = 0u;
  }
}

// The sequence's rows are all done: acceptance in order, then the replacement
// or bonus token; writes the outputs (or hands the sequence to the cluster
// kernel) and re-arms the ticket.
__device__ __noinline__ void kh_finalize(const Params& P, int b, KhShared& S) {
  const int K = P.K, R2 = 2 * K + 1, tid = threadIdx.x;
  const KhRow* rr = P.ws_rowres + (size_t)b * R2;
  const __nv_bfloat16* tgt = static_cast<const __nv_bfloat16*>(P.rows0) + (size_t)b * (K + 1) * P.V;
  const __nv_bfloat16* drf = static_cast<const __nv_bfloat16*>(P.rows1) + (size_t)b * K * P.V;
  KF_MARK(b, 0);
  if (tid < 32) {
    uint32_t f = 0;
    for (int r = tid; r < R2; r += 32) f |= __ldcg(&rr[r].flags);
    if (tid <= K) S.llen[tid] = __ldcg(&rr[tid].pad[1]);
#pragma unroll
    for (int o = 16; o; o >>= 1) f |= __shfl_xor_sync(0xffffffffu, f, o);
    uint32_t ok = 1u;
    bool need = false;
    if (tid < K && !(f & (KH_ERR | KH_BAIL))) {
      const int i = tid;
      const int d = P.dtok[(size_t)b * K + i];
      const KhRow tp = kh_load_row(rr + i), tq = kh_load_row(rr + K + 1 + i);
      const float zp = kh_ldz(P.rows0, (size_t)b * (K + 1) + i, P.V, d);
      const float zq = kh_ldz(P.rows1, (size_t)b * K + i, P.V, d);
      const float p = kh_kept(zp, d, tp.zt, tp.idcut) ? __fmul_rn(kh_w(zp, tp.m, tp.c), tp.invZ) : 0.0f;
      const float qw = __fmul_rn(kh_w(zq, tq.m, tq.c), tq.invZ);
      // d on the draft's cut value with the id split deferred: kept iff fewer
      // than quota tokens on that value precede it (counted below)
      need = tq.idcut == KH_DEFER && zq == tq.zt;
      const float q = kh_kept(zq, d, tq.zt, tq.idcut) ? qw : 0.0f;
      uint32_t ku, kv;
      philox_uniform_bits(P.seed, philox_offset_of(P), (uint32_t)b, (uint32_t)i, &ku, &kv);
      ok = __fmul_rn((float)ku * 5.9604644775390625e-08f, q) < p ? 1u : 0u;
      S.pz[i] = p;
      S.qz[i] = qw;
      S.ku[i] = ku;
      S.flag[i] = ok;
    }
    const uint32_t nm = __ballot_sync(0xffffffffu, need);
    if (tid == 0) {
      S.flags = (int)f;
      S.need = nm;
    }
  }
  __syncthreads();
  const int flags = S.flags;
  for (uint32_t nm = S.need; nm; nm &= nm - 1u) {
    const int i = __ffs(nm) - 1;
    const KhRow tq = kh_load_row(rr + K + 1 + i);
    const int d = P.dtok[(size_t)b * K + i];
    const uint32_t hb = __float_as_uint(tq.zt) >> 16;
    const uint32_t rank = kh_rank_before(reinterpret_cast<const uint4*>(drf + (size_t)i * P.V), d, hb, S);
    if (tid == 0) {
      const float q = rank < tq.pad[0] ? S.qz[i] : 0.0f;
      S.flag[i] = __fmul_rn((float)S.ku[i] * 5.9604644775390625e-08f, q) < S.pz[i] ? 1u : 0u;
    }
  }
  if (tid == 0) {
    int n = K;
    for (int i = 0; i < K; ++i)
      if (!S.flag[i]) {
        n = i;
        break;
      }
    S.nacc = n;
  }
  __syncthreads();
  const int n = S.nacc;
  KF_MARK(b, 1);
  KF_SET(b, 5, n);
  if (flags & KH_BAIL) {
    // the cluster kernel serves the sequence and clears the flag
    if (tid == 0) {
      P.ws_fb[b] = 1u;
      atomicOr(P.ws_work, 1u);
      P.ws_tickets[b] = 0u;
    }
    kh_clear_lists(P, b, S);
    __syncthreads();
    uint4* rz = reinterpret_cast<uint4*>(P.ws_rowres + (size_t)b * R2);
    for (int t = tid; t < 2 * R2; t += KT) rz[t] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  int tok = -1;
  if (!(flags & KH_ERR)) {
    const bool paired = n < K;
    const KhRow tp = kh_load_row(rr + n);
    KhRow tq = paired ? kh_load_row(rr + K + 1 + n) : tp;
    uint32_t ku, kv;
    philox_uniform_bits(P.seed, philox_offset_of(P), (uint32_t)b, (uint32_t)n, &ku, &kv);
    const int nv = P.V / 8;
    const uint4* sp = reinterpret_cast<const uint4*>(tgt + (size_t)n * P.V);
    const uint4* sq = paired ? reinterpret_cast<const uint4*>(drf + (size_t)n * P.V) : sp;
    KhW wq = kh_wof(tq);
    const uint32_t L = tp.pad[1];
    const uint32_t* glist = P.ws_lists + ((size_t)b * (K + 1) + n) * KH_KCAP;
    const unsigned short* zpr = reinterpret_cast<const unsigned short*>(sp);
    const unsigned short* zqr = reinterpret_cast<const unsigned short*>(sq);
    if (L != KH_NOLIST) tok = kh_sample_list(zpr, zqr, glist, (int)L, paired, kh_wof(tp), wq, kv, S);
    else tok = kh_sample(sp, sq, nv, paired, kh_wof(tp), wq, kv, S, b);
    KF_MARK(b, 2);
    KF_SET(b, 4, tok == -2 ? 1 : 0);
    if (tok == -2) {
      // a token of the target's kept set sits on the draft's deferred cut value
      wq.idcut = kh_tie(sq, nv, __float_as_uint(tq.zt) >> 16, (int)tq.pad[0], S);
      if (wq.idcut < 0) tok = -1;
      else if (L != KH_NOLIST) tok = kh_sample_list(zpr, zqr, glist, (int)L, paired, kh_wof(tp), wq, kv, S);
      else tok = kh_sample(sp, sq, nv, paired, kh_wof(tp), wq, kv, S, b);
    }
  }
  if (tid == 0) {
    const bool bad = (flags & KH_ERR) || tok < 0;
    int32_t* ot = P.out_tokens + (size_t)b * (K + 1);
    for (int q = 0; q <= K; ++q)
      ot[q] = bad ? -1 : (q < n ? P.dtok[(size_t)b * K + q] : (q == n ? tok : -1));
    P.out_n[b] = bad ? -1 : n;
    P.ws_tickets[b] = 0u;
  }
  // the call leaves the workspace zeroed
  kh_clear_lists(P, b, S);
  __syncthreads();
  uint4* rz = reinterpret_cast<uint4*>(P.ws_rowres + (size_t)b * R2);
  for (int t = tid; t < 2 * R2; t += KT) rz[t] = make_uint4(0u, 0u, 0u, 0u);
  KF_MARK(b, 3);
}

// Persistent CTAs take rows of the batch's sampled sequences from a work counter
// (sequence-major, so a sequence's rows finish close together and its sampling
// pass finds them in L2). Rows of other sequences are skipped.
__global__ void __launch_bounds__(KT, 2) keyhist_kernel(const Params P, int nitems) {
  uint32_t* kh_hist = kh_dyn;
  __shared__ KhShared S;
  // the cluster kernel may launch now; it waits for this grid before reading
  asm volatile("griddepcontrol.launch_dependents;");
  const int tid = threadIdx.x;
  const int K = P.K, R2 = 2 * K + 1;
  for (int wd = tid; wd < KH_NW; wd += KT) kh_hist[wd] = 0u;
  while (true) {
    if (tid == 0) S.item = (int)atomicAdd(P.ws_fnext, 1u);
    __syncthreads();
    const int item = S.item;
    __syncthreads();
    if (item >= nitems) break;
    const int b = item / R2, r = item - b * R2;
    if (!fast_seq(P, b)) continue;
    KH_MARK(item, 0);
#ifdef SV_TRACE
    if (tid == 0 && item < 8192) {
      uint32_t smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      g_khtrace[item * 8 + 7] = smid;
    }
#endif
    const __nv_bfloat16* row =
        r <= K ? static_cast<const __nv_bfloat16*>(P.rows0) + ((size_t)b * (K + 1) + r) * P.V
               : static_cast<const __nv_bfloat16*>(P.rows1) + ((size_t)b * K + (r - K - 1)) * P.V;
    uint32_t* glist = r <= K ? P.ws_lists + ((size_t)b * (K + 1) + r) * KH_KCAP : nullptr;
    const KhRow res = kh_row(row, P.V, P.temp[b], P.topk[b], P.topp[b], r <= K, kh_hist, S, glist, item);
    KH_MARK(item, 4);
#ifdef SV_TRACE
    if (tid == 0 && item < 8192) g_khtrace[item * 8 + 7] |= (unsigned long long)res.flags << 20;
#endif
    if (tid == 0) {
      uint4* dst = reinterpret_cast<uint4*>(P.ws_rowres + item);
      dst[0] = make_uint4(__float_as_uint(res.zt), __float_as_uint(res.invZ), __float_as_uint(res.m),
                          __float_as_uint(res.c));
      dst[1] = make_uint4((uint32_t)res.idcut, res.flags, res.pad[0], res.pad[1]);
      __threadfence();
      S.last = atomicAdd(&P.ws_tickets[b], 1u) == (unsigned int)(R2 - 1);
      if (S.last) __threadfence();
    }
    __syncthreads();
    if (S.last) {
      KH_MARK(item, 5);
      kh_finalize(P, b, S);
      KH_MARK(item, 6);
    }
    __syncthreads();
  }
  // finish only after greedy_kernel (launched before, possibly still running):
  // whatever waits for this grid then sees both
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the last CTA to leave re-arms the work counter for the next call
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(P.ws_fdone, 1u) == gridDim.x - 1u) {
      *P.ws_fnext = 0u;
      *P.ws_fdone = 0u;
    }
  }
}

// ---------------------------------------------------------- draft sampler
// A row the draft sampler leaves to the cluster kernel (temperature 0, a parameter
// error, or a hand-back) carries this value in out_tokens until that kernel runs.
constexpr int KH_HANDBACK = -2;

// Draft-side sampler for bf16 rows (spec_sample): d ~ q for every row [B][K][V].
// CTAs take rows by a static stride (there is no workspace for a work counter).
// Each row is cut like a target row (window candidates, id split) and sampled in
// the same CTA with the sampling uniform of Philox (b, i): over the kept ids when
// they fit the shared list, else by a full-row inverse CDF.
__global__ void __launch_bounds__(KT, 2) keyhist_sample_kernel(const Params P, int nitems) {
  uint32_t* hist = kh_dyn;
  __shared__ KhShared S;
  const int tid = threadIdx.x;
  for (int wd = tid; wd < KH_NW; wd += KT) hist[wd] = 0u;
  __syncthreads();
  uint32_t* klist = reinterpret_cast<uint32_t*>(kh_blk0());   // kept ids (after the cut)
  const int nv = P.V / 8;
  for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
    const int b = item / P.K, i = item - b * P.K;
    const float T = P.temp[b];
    const bool served = T > 0.0f && T < INFINITY && P.topp[b] > 0.0f && P.topk[b] >= 0 &&
                        __fdiv_rn(KH_LOG2E, T) < 65536.0f;
    if (!served) {
      if (tid == 0) P.out_tokens[item] = KH_HANDBACK;
      continue;
    }
    KH_MARK(item, 0);
    const __nv_bfloat16* row = static_cast<const __nv_bfloat16*>(P.rows0) + (size_t)item * P.V;
    const KhRow res = kh_row(row, P.V, T, P.topk[b], P.topp[b], true, hist, S, klist, item);
    KH_MARK(item, 4);
    int tok;
    if (res.flags & KH_ERR) {
      tok = -1;
    } else if (res.flags & KH_BAIL) {
      tok = KH_HANDBACK;
    } else {
      uint32_t ku, kv;
      philox_uniform_bits(P.seed, philox_offset_of(P), (uint32_t)b, (uint32_t)i, &ku, &kv);
      const KhW w = kh_wof(res);
      if (res.pad[1] != KH_NOLIST) {
        const unsigned short* zr = reinterpret_cast<const unsigned short*>(row);
        tok = kh_sample_list(zr, zr, klist, (int)res.pad[1], false, w, w, kv, S);   // scratch: the histogram
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(row);
        tok = kh_sample(src, src, nv, false, w, w, kv, S, -1);
      }
      if (tok < 0) tok = -1;
    }
    KH_MARK(item, 5);
    if (tid == 0) P.out_tokens[item] = tok;
    __syncthreads();
  }
}

// ------------------------------------------------- truncated probabilities
// A row spec_truncated_probs leaves to the cluster kernel carries this bit pattern
// in out_probs[row][0] (a NaN payload no kernel writes otherwise).
constexpr uint32_t KH_PROBS_HANDBACK = 0x7FC0BEEFu;

// spec_truncated_probs for bf16 rows through the per-row code of the sampled
// verify path (kh_row: stream, sparse or full histogram, exact fixed-point cut and
// normaliser, id split), then p(x) = kh_w(z, m, c) * 2^44 / Z for kept tokens, as
// kh_elem computes it for the verify's acceptance test and inverse CDF. Rows
// [R][V]; temperature-0 rows, parameter errors and hand-backs are marked for the
// cluster kernel; data errors write NaN to the row.
__global__ void __launch_bounds__(KT, 2) keyhist_probs_kernel(const Params P, int nitems) {
  uint32_t* hist = kh_dyn;
  __shared__ KhShared S;
  const int tid = threadIdx.x;
  for (int wd = tid; wd < KH_NW; wd += KT) hist[wd] = 0u;
  __syncthreads();
  uint32_t* klist = reinterpret_cast<uint32_t*>(kh_blk0());
  for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
    const float T = P.temp[item];
    float* out = P.out_probs + (size_t)item * P.V;
    const bool served = T > 0.0f && T < INFINITY && P.topp[item] > 0.0f && P.topk[item] >= 0 &&
                        __fdiv_rn(KH_LOG2E, T) < 65536.0f;
    if (!served) {
      if (tid == 0) out[0] = __uint_as_float(KH_PROBS_HANDBACK);
      continue;
    }
    const __nv_bfloat16* row = static_cast<const __nv_bfloat16*>(P.rows0) + (size_t)item * P.V;
    const KhRow res = kh_row(row, P.V, T, P.topk[item], P.topp[item], true, hist, S, klist, item);
    if (res.flags & KH_BAIL) {
      if (tid == 0) out[0] = __uint_as_float(KH_PROBS_HANDBACK);
    } else if (res.flags & KH_ERR) {
      for (int x = tid; x < P.V; x += KT) out[x] = __uint_as_float(0x7fc00000u);
    } else {
      const unsigned short* zr = reinterpret_cast<const unsigned short*>(row);
      for (int x = tid; x < P.V; x += KT) {
        const float z = __uint_as_float((uint32_t)__ldg(zr + x) << 16);
        out[x] = kh_kept(z, x, res.zt, res.idcut) ? __fmul_rn(kh_w(z, res.m, res.c), res.invZ) : 0.0f;
      }
    }
    __syncthreads();
  }
}

}  // namespace sv
