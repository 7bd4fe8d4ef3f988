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
constexpr size_t KH_SMEM = (size_t)KH_NW * 4;
constexpr float KH_LOG2E = 1.44269504088896341f;

constexpr uint32_t KH_ERR = 1u, KH_BAIL = 2u;

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
  uint32_t flag[64];
};

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

// Counts the 8 logits of one vector and folds them into the running maximum.
__device__ __forceinline__ void kh_count8(uint32_t* hist, const uint4& w, __nv_bfloat162& m2) {
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
  m2 = __hmax2(__hmax2(m2, a), __hmax2(__hmax2(b, c), d));
}

// Streams one row (nv 16-byte vectors) into the histogram; returns this
// thread's maximum (NaN is ignored here: NaN bins are checked afterwards).
__device__ __forceinline__ float kh_stream(const uint4* src, int nv, uint32_t* hist) {
  const int tid = threadIdx.x;
  uint4 buf[KH_PF];
#pragma unroll
  for (int p = 0; p < KH_PF; ++p) {
    const int q = tid + p * KT;
    if (q < nv) buf[p] = kh_ld(src + q);
  }
  __nv_bfloat162 m2 = __halves2bfloat162(__ushort_as_bfloat16((unsigned short)0xFF80u),
                                         __ushort_as_bfloat16((unsigned short)0xFF80u));
  for (int q0 = tid; q0 < nv; q0 += KH_PF * KT) {
#pragma unroll
    for (int p = 0; p < KH_PF; ++p) {
      const int q = q0 + p * KT;
      if (q < nv) {
        const uint4 w = buf[p];
        const int qn = q + KH_PF * KT;
        if (qn < nv) buf[p] = kh_ld(src + qn);
        kh_count8(hist, w, m2);
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

// The id of the q-th (1-based) token, in id order, whose logit pattern is hb.
// Each warp counts a contiguous id range; the warp holding the q-th match
// locates it with a lane-order scan. -1 if there are fewer than q matches.
__device__ __noinline__ int kh_tie(const uint4* src, int nv, uint32_t hb, int q, KhShared& S) {
  const int w = warp_id(), l = lane_id();
  const int cw = (nv + KWARP - 1) / KWARP;
  const int a0 = min(w * cw, nv), a1 = min(a0 + cw, nv);
  uint32_t n = 0;
  for (int v = a0 + l; v < a1; v += 32) n += __popc(kh_match8(kh_ld_l2(src + v), hb));
  n = warp_sum(n);
  if (l == 0) S.s32[w] = n;
  if (threadIdx.x == 0) S.idcut = -1;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t acc = 0;
    S.wq = -1;
    for (int i = 0; i < KWARP; ++i) {
      if (acc + S.s32[i] >= (uint32_t)q) {
        S.wq = i;
        S.rq = q - (int)acc;
        break;
      }
      acc += S.s32[i];
    }
  }
  __syncthreads();
  if (w == S.wq) {
    int r = S.rq;
    for (int v0 = a0; v0 < a1; v0 += 32) {
      const int v = v0 + l;
      const uint32_t mk = v < a1 ? kh_match8(kh_ld_l2(src + v), hb) : 0u;
      const int cnt = __popc(mk);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (l >= o) incl += t;
      }
      const int excl = incl - cnt;
      const uint32_t bal = __ballot_sync(0xffffffffu, excl < r && r <= incl);
      if (bal) {
        if (l == __ffs(bal) - 1) {
          int need = r - excl;
          for (int e = 0; e < 8; ++e)
            if ((mk >> e) & 1u)
              if (--need == 0) {
                S.idcut = v * 8 + e;
                break;
              }
        }
        break;
      }
      r -= __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  return S.idcut;
}

// Weight of bin idx in fixed point (0 for -inf; NaN / +inf bins never get here).
__device__ __forceinline__ unsigned long long kh_binw(int idx, float m, float c) {
  return idx > KH_NINF ? kh_fix(kh_value(idx), m, c) : 0ull;
}

// One row: histogram, maximum, normaliser, top-k / top-p cut and the id split of
// a partial cut bin. Leaves the histogram zeroed. The result is returned in
// every thread.
__device__ __noinline__ KhRow kh_row(const __nv_bfloat16* row, int V, float T, int k, float topP,
                                     uint32_t* hist, KhShared& S) {
  const int tid = threadIdx.x, l = lane_id(), w = warp_id();
  const int nv = V / 8;
  const uint4* src = reinterpret_cast<const uint4*>(row);
  float mt = kh_stream(src, nv, hist);
#pragma unroll
  for (int o = 16; o; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
  if (l == 0) S.fmax[w] = mt;
  __syncthreads();                              // the histogram is complete
  float m = S.fmax[0];
#pragma unroll
  for (int i = 1; i < KWARP; ++i) m = fmaxf(m, S.fmax[i]);
  const float c = __fdiv_rn(KH_LOG2E, T);

  // sweep: counts and fixed-point masses of this thread's bins
  const int w0 = min(tid * KH_WPT, KH_NW), w1 = min(w0 + KH_WPT, KH_NW);
  uint32_t cnt = 0, bad = 0;
  unsigned long long mass = 0;
  for (int wd = w0; wd < w1; ++wd) {
    const uint32_t x = hist[wd];
    if (x == 0u) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t cb = h ? x >> 16 : x & 0xFFFFu;
      if (cb == 0u) continue;
      const int idx = 2 * wd + h;
      cnt += cb;
      if (idx < KH_NINF || idx >= KH_PINF) bad = 1u;
      else mass += (unsigned long long)cb * kh_binw(idx, m, c);
    }
  }
  const int anyb = __syncthreads_or((int)bad);
  uint32_t ctot;
  const uint32_t cab = kh_above<uint32_t>(cnt, S.s32, &ctot);
  unsigned long long Ztot;
  const unsigned long long mab = kh_above<unsigned long long>(mass, S.s64, &Ztot);

  KhRow res;
  res.m = m;
  res.c = c;
  res.zt = -INFINITY;
  res.idcut = V;
  res.invZ = 0.0f;
  res.flags = 0u;
  res.pad[0] = res.pad[1] = 0u;
  if (anyb || !(m > -INFINITY)) res.flags = KH_ERR;
  else if (ctot != (uint32_t)V) res.flags = KH_BAIL;
  const bool topk = k > 0 && k < V;
  const bool topp = topP < 1.0f;
  if (res.flags == 0u && topk) {
    // the bin holding the k-th token in (logit desc, id asc) order
    if (cab < (uint32_t)k && (uint32_t)k <= cab + cnt) {
      uint32_t acc = cab;
      unsigned long long M = mab;
      for (int wd = w1 - 1; wd >= w0; --wd) {
        const uint32_t x = hist[wd];
        if (x == 0u) continue;
        bool done = false;
#pragma unroll
        for (int h = 1; h >= 0; --h) {
          const uint32_t cb = h ? x >> 16 : x & 0xFFFFu;
          if (cb == 0u || done) continue;
          const int idx = 2 * wd + h;
          const unsigned long long W = kh_binw(idx, m, c);
          if (acc + cb >= (uint32_t)k) {
            S.kbin = idx;
            S.kq = k - (int)acc;
            S.Mk = M;
            S.Wk = W;
            S.ccnt = (int)cb;
            done = true;
          } else {
            acc += cb;
            M += (unsigned long long)cb * W;
          }
        }
        if (done) break;
      }
    }
    __syncthreads();
  }
  if (res.flags == 0u && (topk || topp)) {
    const unsigned long long ZL1 = topk ? S.Mk + (unsigned long long)S.kq * S.Wk : Ztot;
    if (topp) {
      // the bin where the exclusive mass first exceeds Y = the largest integer
      // below P * Z(L1); tokens with exclusive mass <= Y are kept
      const unsigned long long Y = mass_threshold(topP, ZL1);
      if (mab <= Y && Y < mab + mass) {
        unsigned long long M = mab;
        for (int wd = w1 - 1; wd >= w0; --wd) {
          const uint32_t x = hist[wd];
          if (x == 0u) continue;
          bool done = false;
#pragma unroll
          for (int h = 1; h >= 0; --h) {
            const uint32_t cb = h ? x >> 16 : x & 0xFFFFu;
            if (cb == 0u || done) continue;
            const int idx = 2 * wd + h;
            const unsigned long long W = kh_binw(idx, m, c);
            if (M + (unsigned long long)cb * W > Y) {
              S.cbin = idx;
              S.cq = (int)((Y - M) / W) + 1;
              S.Mcut = M;
              S.Wcut = W;
              S.ccnt = (int)cb;
              done = true;
            } else {
              M += (unsigned long long)cb * W;
            }
          }
          if (done) break;
        }
      }
    } else if (tid == 0) {
      S.cbin = S.kbin;
      S.cq = S.kq;
      S.Mcut = S.Mk;
      S.Wcut = S.Wk;
    }
    __syncthreads();
  }
  // the histogram is not read again for this row
  for (int wd = w0; wd < w1; ++wd) hist[wd] = 0u;
  if (res.flags != 0u) return res;

  unsigned long long Zk = Ztot;
  if (topk || topp) {
    const int cbin = S.cbin, q = S.cq, ccnt = S.ccnt;
    Zk = S.Mcut + (unsigned long long)q * S.Wcut;
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
      const uint32_t hb = __float_as_uint(kh_value(cbin)) >> 16;
      res.zt = kh_value(cbin);
      res.idcut = kh_tie(src, nv, hb, q, S);
      if (res.idcut < 0) res.flags = KH_BAIL;
    }
  }
  res.invZ = __fdiv_rn(17592186044416.0f, (float)Zk);   // 2^44 / Z
  return res;
}

// Sampling weights of one token: r = (p - q)+ and p, both 0 outside the
// target's kept set (probabilities in fp32, as 2^44-frame weights times 1/Z).
__device__ __forceinline__ void kh_elem(float zp, float zq, int id, bool paired, const KhRow& tp,
                                        const KhRow& tq, float* r, float* p) {
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

// Fixed-point (2^-40) residual and target masses of the 8 tokens of vector v.
__device__ __forceinline__ void kh_vec_sums(const uint4* sp, const uint4* sq, int v, bool paired,
                                            const KhRow& tp, const KhRow& tq,
                                            unsigned long long* R, unsigned long long* Pm) {
  const uint4 a = kh_ld_l2(sp + v);
  const uint32_t as[4] = {a.x, a.y, a.z, a.w};
  // cheap test first: most tokens of a peaked target row are outside its kept set
  bool any = false;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    any |= kh_kept(kh_lo(as[k]), v * 8 + 2 * k, tp.zt, tp.idcut) |
           kh_kept(kh_hi(as[k]), v * 8 + 2 * k + 1, tp.zt, tp.idcut);
  *R = 0ull;
  *Pm = 0ull;
  if (!any) return;
  uint4 b = make_uint4(0u, 0u, 0u, 0u);
  if (paired) b = kh_ld_l2(sq + v);
  const uint32_t bs[4] = {b.x, b.y, b.z, b.w};
  unsigned long long ra = 0, pa = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float r, p;
    kh_elem(kh_lo(as[k]), kh_lo(bs[k]), v * 8 + 2 * k, paired, tp, tq, &r, &p);
    ra += fixr(r);
    pa += fixr(p);
    kh_elem(kh_hi(as[k]), kh_hi(bs[k]), v * 8 + 2 * k + 1, paired, tp, tq, &r, &p);
    ra += fixr(r);
    pa += fixr(p);
  }
  *R = ra;
  *Pm = pa;
}

// Inverse CDF in token-id order over (p - q)+ (paired) or p: the smallest id j
// whose running sum S_j satisfies S_j * 2^24 > kv * S (S the total); when the
// residual mass is 0 the target p is used. -1 if no token qualifies.
__device__ __noinline__ int kh_sample(const uint4* sp, const uint4* sq, int nv, bool paired,
                                      const KhRow& tp, const KhRow& tq, uint32_t kv,
                                      KhShared& S) {
  const int w = warp_id(), l = lane_id();
  const int cw = (nv + KWARP - 1) / KWARP;
  const int a0 = min(w * cw, nv), a1 = min(a0 + cw, nv);
  unsigned long long R = 0, Pm = 0;
  for (int v = a0 + l; v < a1; v += 32) {
    unsigned long long r, p;
    kh_vec_sums(sp, sq, v, paired, tp, tq, &r, &p);
    R += r;
    Pm += p;
  }
  R = warp_sum(R);
  Pm = warp_sum(Pm);
  if (l == 0) {
    S.s64[w] = R;
    S.s64b[w] = Pm;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long SR = 0, SP = 0;
    for (int i = 0; i < KWARP; ++i) {
      SR += S.s64[i];
      SP += S.s64b[i];
    }
    const bool useR = SR > 0ull;
    const unsigned long long St = useR ? SR : SP;
    unsigned long long acc = 0;
    S.wq = -1;
    for (int i = 0; i < KWARP; ++i) {
      const unsigned long long own = useR ? S.s64[i] : S.s64b[i];
      if (mul_gt(acc + own, 1ull << 24, kv, St)) {
        S.wq = i;
        break;
      }
      acc += own;
    }
    S.acc = acc;
    S.useR = useR;
    S.Mcut = St;
    S.tok = -1;
  }
  __syncthreads();
  if (w == S.wq) {
    const bool useR = S.useR != 0;
    const unsigned long long St = S.Mcut;
    unsigned long long acc = S.acc;
    for (int v0 = a0; v0 < a1; v0 += 32) {
      const int v = v0 + l;
      unsigned long long r = 0, p = 0;
      if (v < a1) kh_vec_sums(sp, sq, v, paired, tp, tq, &r, &p);
      const unsigned long long own = useR ? r : p;
      unsigned long long incl = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (l >= o) incl += t;
      }
      const bool hit = v < a1 && mul_gt(acc + incl, 1ull << 24, kv, St);
      const uint32_t bal = __ballot_sync(0xffffffffu, hit);
      if (bal) {
        if (l == __ffs(bal) - 1) {
          // walk this vector's tokens in id order
          const uint4 a = kh_ld_l2(sp + v);
          uint4 b = make_uint4(0u, 0u, 0u, 0u);
          if (paired) b = kh_ld_l2(sq + v);
          const uint32_t as[4] = {a.x, a.y, a.z, a.w}, bs[4] = {b.x, b.y, b.z, b.w};
          unsigned long long run = acc + incl - own;
          int tok = -1;
          for (int e = 0; e < 8 && tok < 0; ++e) {
            const uint32_t xa = as[e >> 1], xb = bs[e >> 1];
            const float zp = (e & 1) ? kh_hi(xa) : kh_lo(xa);
            const float zq = (e & 1) ? kh_hi(xb) : kh_lo(xb);
            float rr, pp;
            kh_elem(zp, zq, v * 8 + e, paired, tp, tq, &rr, &pp);
            run += fixr(useR ? rr : pp);
            if (mul_gt(run, 1ull << 24, kv, St)) tok = v * 8 + e;
          }
          S.tok = tok;
        }
        break;
      }
      acc += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  return S.tok;
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

// The sequence's rows are all done: acceptance in order, then the replacement
// or bonus token; writes the outputs (or hands the sequence to the cluster
// kernel) and re-arms the ticket.
__device__ __noinline__ void kh_finalize(const Params& P, int b, KhShared& S) {
  const int K = P.K, R2 = 2 * K + 1, tid = threadIdx.x;
  const KhRow* rr = P.ws_rowres + (size_t)b * R2;
  if (tid < 32) {
    uint32_t f = 0;
    for (int r = tid; r < R2; r += 32) f |= __ldcg(&rr[r].flags);
#pragma unroll
    for (int o = 16; o; o >>= 1) f |= __shfl_xor_sync(0xffffffffu, f, o);
    uint32_t ok = 1u;
    if (tid < K && !(f & (KH_ERR | KH_BAIL))) {
      const int i = tid;
      const int d = P.dtok[(size_t)b * K + i];
      const KhRow tp = kh_load_row(rr + i), tq = kh_load_row(rr + K + 1 + i);
      const float zp = kh_ldz(P.rows0, (size_t)b * (K + 1) + i, P.V, d);
      const float zq = kh_ldz(P.rows1, (size_t)b * K + i, P.V, d);
      const float p = kh_kept(zp, d, tp.zt, tp.idcut) ? __fmul_rn(kh_w(zp, tp.m, tp.c), tp.invZ) : 0.0f;
      const float q = kh_kept(zq, d, tq.zt, tq.idcut) ? __fmul_rn(kh_w(zq, tq.m, tq.c), tq.invZ) : 0.0f;
      uint32_t ku, kv;
      philox_uniform_bits(P.seed, P.offset, (uint32_t)b, (uint32_t)i, &ku, &kv);
      ok = __fmul_rn((float)ku * 5.9604644775390625e-08f, q) < p ? 1u : 0u;
    }
    const uint32_t rej = __ballot_sync(0xffffffffu, tid < K && !ok);
    if (tid == 0) {
      S.flags = (int)f;
      S.nacc = rej ? __ffs(rej) - 1 : K;
    }
  }
  __syncthreads();
  const int flags = S.flags, n = S.nacc;
  if (flags & KH_BAIL) {
    // the cluster kernel serves the sequence and clears the flag
    if (tid == 0) {
      P.ws_fb[b] = 1u;
      atomicOr(P.ws_work, 1u);
      P.ws_tickets[b] = 0u;
    }
    uint4* rz = reinterpret_cast<uint4*>(P.ws_rowres + (size_t)b * R2);
    for (int t = tid; t < 2 * R2; t += KT) rz[t] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  int tok = -1;
  if (!(flags & KH_ERR)) {
    const bool paired = n < K;
    const KhRow tp = kh_load_row(rr + n);
    const KhRow tq = paired ? kh_load_row(rr + K + 1 + n) : tp;
    uint32_t ku, kv;
    philox_uniform_bits(P.seed, P.offset, (uint32_t)b, (uint32_t)n, &ku, &kv);
    const int nv = P.V / 8;
    const uint4* sp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(P.rows0) +
                                                     ((size_t)b * (K + 1) + n) * P.V);
    const uint4* sq = paired ? reinterpret_cast<const uint4*>(
                                   static_cast<const __nv_bfloat16*>(P.rows1) + ((size_t)b * K + n) * P.V)
                             : sp;
    tok = kh_sample(sp, sq, nv, paired, tp, tq, kv, S);
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
  uint4* rz = reinterpret_cast<uint4*>(P.ws_rowres + (size_t)b * R2);
  for (int t = tid; t < 2 * R2; t += KT) rz[t] = make_uint4(0u, 0u, 0u, 0u);
}

// Persistent CTAs take rows of the batch's sampled sequences from a work counter
// (sequence-major, so a sequence's rows finish close together and its sampling
// pass finds them in L2). Rows of other sequences are skipped.
__global__ void __launch_bounds__(KT, 2) keyhist_kernel(const Params P, int nitems) {
  extern __shared__ __align__(16) uint32_t kh_hist[];
  __shared__ KhShared S;
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
    const __nv_bfloat16* row =
        r <= K ? static_cast<const __nv_bfloat16*>(P.rows0) + ((size_t)b * (K + 1) + r) * P.V
               : static_cast<const __nv_bfloat16*>(P.rows1) + ((size_t)b * K + (r - K - 1)) * P.V;
    const KhRow res = kh_row(row, P.V, P.temp[b], P.topk[b], P.topp[b], kh_hist, S);
    if (tid == 0) {
      uint4* dst = reinterpret_cast<uint4*>(P.ws_rowres + item);
      dst[0] = make_uint4(__float_as_uint(res.zt), __float_as_uint(res.invZ), __float_as_uint(res.m),
                          __float_as_uint(res.c));
      dst[1] = make_uint4((uint32_t)res.idcut, res.flags, 0u, 0u);
      __threadfence();
      S.last = atomicAdd(&P.ws_tickets[b], 1u) == (unsigned int)(R2 - 1);
      if (S.last) __threadfence();
    }
    __syncthreads();
    if (S.last) kh_finalize(P, b, S);
    __syncthreads();
  }
  // the last CTA to leave re-arms the work counter for the next call
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(P.ws_fdone, 1u) == gridDim.x - 1u) {
      *P.ws_fnext = 0u;
      *P.ws_fdone = 0u;
    }
  }
}

}  // namespace sv
