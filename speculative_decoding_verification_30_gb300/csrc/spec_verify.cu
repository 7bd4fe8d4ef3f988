// spec_verify.cu -- verify-and-sample kernels for GB300 (sm_103a) and the C ABI.
//
// Work decomposition. A "unit" is one (sequence b, position i) pair, i in
// [0, K]: for i < K it owns target row i and draft row i, for i == K the
// target row K (bonus position). One thread-block cluster of C CTAs serves one
// unit; CTA c holds the vocabulary slice [c*slice, (c+1)*slice) of the unit's
// rows in shared memory, loaded once from HBM by bulk copies (TMA engine).
// Every later pass reads shared memory only; CTAs combine partial results
// through distributed shared memory (DSMEM).
//
// Method (pages cited in include/spec_verify.h): temperature scaling, matched
// top-k / top-p truncation of target and draft, acceptance with min(1, p/q) in
// order, replacement from (p - q)+ or the bonus token from p_K, greedy
// argmax-prefix matching at temperature 0.
//
// Passes per row of a sampling unit:
//   A  row maximum (NaN/+inf check), argmax, per-thread maxima.       [X1]
//   B  top-k rows: collect the tokens that can be in the top k (at or above
//      the largest per-CTA k-th largest per-thread maximum: each CTA alone
//      holds k tokens that large). No exponentials.
//      top-p rows: weights e = exp((z - m)/T) once per token; exact mass of
//      the head (tokens within 8 nats of the maximum, listed); private
//      per-thread mass/count histograms of the tail in 1-nat distance bins
//      (no shared-memory atomics: every thread owns its counters).     [X2]
//   R  (top-p rows whose cut lies in the tail) refinement: the bin holding
//      the cut is split into 16 sub-bins, touching only tokens inside it,
//      until the range holding the cut is small enough to list.        [X3..]
//   L  list the tokens of that range.
//   S  the listed tokens of every CTA are pushed to CTA 0, which sorts them
//      by (logit desc, id asc) and finds the cut exactly.          [push, res]
//   then the probabilities of the draft token, and the inverse-CDF scan of
//   (p - q)+ (or p) in token-id order across the cluster.              [CDF]
// Rows where the lists would not fit take the general path: a distributed
// radix selection over the whole slice (slower, same results).
//
// Sums: weights are converted to fixed point floor(e * 2^S), S = 63 -
// ceil(log2 V); histogram masses and the normaliser are integer sums of
// per-thread partial sums. The inverse-CDF decision C_j * 2^24 > k_v * S is
// taken exactly on 64-bit integers.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/spec_verify.h"
#include "sv_device.cuh"

namespace sv {

// Phase timestamps for profiling builds (-DSV_TRACE): CTA rank 0, thread 0 of
// the first 256 units records %globaltimer at each marker. Compiled out otherwise.
#ifdef SV_TRACE
__device__ unsigned long long g_trace[256 * 16];
#define SV_MARK(k)                                                              \
  do {                                                                         \
    if (threadIdx.x == 0 && cluster_rank() == 0 && unit < 256)                 \
      g_trace[unit * 16 + (k)] = global_timer_ns();                            \
  } while (0)
#else
#define SV_MARK(k) ((void)0)
#endif

enum Mode { MODE_VERIFY = 0, MODE_PROBS = 1, MODE_SAMPLE = 2 };

struct Params {
  const void* rows0;        // VERIFY: target [B,K+1,V]; PROBS/SAMPLE: logits
  const void* rows1;        // VERIFY: draft [B,K,V] (may be null)
  const int32_t* dtok;      // [B,K]
  const float* temp;
  const int32_t* topk;
  const float* topp;
  uint64_t seed, offset;
  int B, K, V;
  int nunits;
  int slice;                // elements per CTA per row (multiple of 16)
  int ept;                  // elements per thread (contiguous range)
  int bulk_ok;              // rows are 16-byte aligned: use bulk copies
  int nlev;                 // radix levels of the general path: 2 (bf16) or 4 (fp32)
  uint32_t keymask;         // key bits that vary: 0xffff0000 for bf16 logits, all for fp32
  float fix_scale;          // 2^S
  int32_t* out_tokens;
  int32_t* out_n;
  float* out_probs;
  unsigned long long* ws_units;  // per unit: bit 0..31 token, bit 32 flag, bit 33 error
  unsigned int* ws_tickets;      // per sequence
  unsigned int* ws_error;        // sticky: bit 0 = a bulk copy did not complete in time
};

constexpr uint32_t KEY_ALL = 0u;          // threshold that admits every token
constexpr int NO_TIE = 0x7fffffff;        // tie id admitting the whole tie group
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr float DHEAD = 8.0f;             // head: within 8 nats of the row maximum
constexpr int NB = 16;                    // bins per histogram level
constexpr int NBH = NB + 1;               // level 0 adds a bin for >= 16 nats beyond the head
constexpr int LCAP = 512;                 // per-CTA list capacity (entries per row)
constexpr int GCAP = 1024;                // entries per row gathered at the selecting CTA
constexpr int MAXLEV = 5;                 // histogram levels before the general path

enum RowMode { RM_FULL = 0, RM_TOPK = 1, RM_TOPP = 2 };
enum Need { ND_DONE = 0, ND_REFINE = 1, ND_LIST = 2, ND_GENERAL = 3, ND_TIE = 4 };

// Per-row state; identical in every CTA of the cluster after each exchange.
struct RowK {
  RowW w;
  int argmax;
  int bad;
  int mode;
  int kk;                      // k' (top-k count; V when off)
  float topp;
  uint32_t tau;                // top-k list admission: key >= tau
  int lev;                     // level of the current range (-1: head / top-k list)
  int q;                       // index of the current range at that level
  int need;
  int pad;
  unsigned long long Z;        // total mass (top-p and full-support rows)
  unsigned long long Zh;       // head mass (top-p rows)
  unsigned long long above;    // mass strictly above the current range
  double X;                    // top-p target mass (fixed-point units)
  uint32_t thr;                // result: kept iff key > thr or (key == thr and id <= tie)
  int tie;
  unsigned long long ZL;       // result: kept mass
  unsigned int jt;             // tie group: members to keep (ND_TIE)
  unsigned int rc[16];         // per-CTA entries of the list being gathered
};

struct XA {                    // X1 payload per row
  float best;
  int best_id;
  int bad;
  uint32_t kth;
};

struct XB {                    // pass-B / refinement payload per row
  unsigned long long zh, zt;
  unsigned int lcnt;
  unsigned int kmin, kmax;     // key range of the tokens in the refined range
  unsigned int pad;
  unsigned long long hm[NBH];
  unsigned int hc[NBH];
};

struct Work {
  unsigned long long mbar;
  unsigned long long pad0;
  XA xa[2];
  XB xb[2][2];                              // [buffer][row]
  RowK rk[2];
  unsigned long long xs[2][2];              // [buffer][slot] small exchanges
  unsigned long long scan64[NWARP];
  unsigned int scan32[NWARP];
  unsigned int lcnt[2];
  unsigned int kthh[2][256];
  int bi[8];
  unsigned long long bu[4];
  uint32_t res_thr[2];
  int res_tie[2];
  unsigned long long res_zl[2];
  int res_fail[2];
  uint16_t list[2][LCAP];
  union {
    struct {
      float pmass[NBH][NT];                 // private per-thread histograms
      uint8_t pcnt[NBH][NT];
    } ph;
    unsigned long long g[2][GCAP];          // gathered entries at the selecting CTA
    struct {                                // general path
      unsigned long long hmass[2][2][256];
      unsigned int hcnt[2][2][256];
      unsigned long long gmass[2][256];
      unsigned int gcnt[2][256];
    } gp;
  } u;
};

// Order key restricted to the bits a logit of this dtype can set. For bf16 the
// low 16 bits of okey() are all zeros (positive) or all ones (negative), so
// they are dropped; radix levels then build exactly these masked keys.
__device__ __forceinline__ uint32_t mkey(float z, uint32_t mask) { return okey(z) & mask; }
// Float value of a masked key (inverse of mkey on values of the dtype).
__device__ __forceinline__ float mkey_to_float(uint32_t k, uint32_t mask) {
  return key_to_float((k & 0x80000000u) ? k : (k | ~mask));
}

template <typename DT>
__device__ __forceinline__ float ld_peer_logit(uint32_t local_base, int j, uint32_t rank);
template <>
__device__ __forceinline__ float ld_peer_logit<float>(uint32_t local_base, int j, uint32_t rank) {
  uint32_t a, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local_base + 4u * j), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return __uint_as_float(v);
}
template <>
__device__ __forceinline__ float ld_peer_logit<__nv_bfloat16>(uint32_t local_base, int j,
                                                              uint32_t rank) {
  uint32_t a;
  uint16_t v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local_base + 2u * j), "r"(rank));
  asm volatile("ld.shared::cluster.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
  return __uint_as_float(((uint32_t)v) << 16);
}

__device__ __forceinline__ float pow16(int l) {
  return __int_as_float((127 + 4 * l) << 23);   // 16^l, exact
}
// Distance beyond the head in temperature-scaled nats, clamped at 0. Every
// pass uses this same expression, so bin membership is consistent.
__device__ __forceinline__ float tail_dist(float z, const RowW& w) {
  return fmaxf(fmaf(w.m - z, w.invT, -DHEAD), 0.0f);
}

// ------------------------------------------------------------------------
// k-th largest of the CTA's per-thread maxima (block radix select on keys).
// Returns KEY_ALL when fewer than k threads hold a token.
__device__ uint32_t block_kth_largest(uint32_t key, bool valid, int k, unsigned int* hist,
                                      unsigned int* scratch, int nlev) {
  uint32_t prefix = 0, mask = 0;
  int need = k;
  for (int lev = 0; lev < nlev; ++lev) {
    const int shift = 24 - 8 * lev;
    for (int t = threadIdx.x; t < 256; t += NT) hist[t] = 0;
    __syncthreads();
    if (valid && (key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    __syncthreads();
    if (warp_id() == 0) {
      const int l = lane_id();
      unsigned int c[8], s = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        c[q] = hist[255 - (8 * l + q)];
        s += c[q];
      }
      unsigned int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        unsigned int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (l >= o) incl += t;
      }
      const unsigned int excl = incl - s;
      const unsigned int total = __shfl_sync(0xffffffffu, incl, 31);
      int digit = -1;
      unsigned int above = 0;
      if ((int)total >= need && (int)excl < need && (int)incl >= need) {
        unsigned int run = excl;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (digit < 0 && (int)(run + c[q]) >= need) {
            digit = 255 - (8 * l + q);
            above = run;
          }
          run += c[q];
        }
      }
      const unsigned int who = __ballot_sync(0xffffffffu, digit >= 0);
      if (who == 0) {
        if (l == 0) scratch[0] = 0xffffffffu;
      } else {
        const int src = __ffs(who) - 1;
        digit = __shfl_sync(0xffffffffu, digit, src);
        above = __shfl_sync(0xffffffffu, above, src);
        if (l == 0) {
          scratch[0] = (unsigned int)digit;
          scratch[1] = above;
        }
      }
    }
    __syncthreads();
    const unsigned int dg = scratch[0];
    const unsigned int ab = scratch[1];
    __syncthreads();
    if (dg == 0xffffffffu) return KEY_ALL;
    prefix |= dg << shift;
    mask |= 255u << shift;
    need -= (int)ab;
  }
  return prefix;
}

// ------------------------------------------------------------------------
// General path: digit where the cumulative (from the top) count or mass of a
// cluster-wide 256-bin histogram first reaches the target (warp-level).
struct DigitPick {
  int digit;
  unsigned int cnt_above;
  unsigned long long mass_above;
};

__device__ DigitPick pick_digit(const unsigned int* gcnt, const unsigned long long* gmass,
                                bool by_mass, unsigned long long need_cnt, double need_mass) {
  const int l = lane_id();
  unsigned int c[8];
  unsigned long long w[8];
  unsigned long long sc = 0, sw = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int dg = 255 - (8 * l + q);
    c[q] = gcnt[dg];
    w[q] = gmass[dg];
    sc += c[q];
    sw += w[q];
  }
  unsigned long long ic = sc, iw = sw;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned long long tc = __shfl_up_sync(0xffffffffu, ic, o);
    unsigned long long tw = __shfl_up_sync(0xffffffffu, iw, o);
    if (l >= o) {
      ic += tc;
      iw += tw;
    }
  }
  unsigned long long rc = ic - sc, rw = iw - sw;
  int digit = -1;
  unsigned long long ac = 0, aw = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const unsigned long long nc = rc + c[q], nw = rw + w[q];
    const bool hit = by_mass ? ((double)nw >= need_mass) : (nc >= need_cnt);
    if (digit < 0 && hit) {
      digit = 255 - (8 * l + q);
      ac = rc;
      aw = rw;
    }
    rc = nc;
    rw = nw;
  }
  const unsigned int who = __ballot_sync(0xffffffffu, digit >= 0);
  DigitPick p;
  if (who == 0) {              // target beyond the total: take the smallest non-empty digit
    const unsigned long long tc = __shfl_sync(0xffffffffu, ic, 31);
    const unsigned long long tw = __shfl_sync(0xffffffffu, iw, 31);
    int lowest = -1;
    for (int dg = 0; dg < 256; ++dg)
      if (gcnt[dg] != 0) {
        lowest = dg;
        break;
      }
    p.digit = lowest < 0 ? 0 : lowest;
    p.cnt_above = (unsigned int)(tc - (lowest < 0 ? 0 : gcnt[lowest]));
    p.mass_above = tw - (lowest < 0 ? 0 : gmass[lowest]);
    return p;
  }
  const int src = __ffs(who) - 1;
  p.digit = __shfl_sync(0xffffffffu, digit, src);
  p.cnt_above = (unsigned int)__shfl_sync(0xffffffffu, ac, src);
  p.mass_above = __shfl_sync(0xffffffffu, aw, src);
  return p;
}

// Publishes one unit's result; the last of the K+1 units of sequence b writes
// the sequence's outputs and re-arms the ticket (leaving the workspace zeroed).
__device__ void publish_unit(const Params& P, int unit, int b, int token, bool flag, bool err) {
  P.ws_units[unit] = (unsigned long long)(uint32_t)token | ((unsigned long long)flag << 32) |
                     ((unsigned long long)err << 33);
  __threadfence();
  const unsigned int old = atomicAdd(&P.ws_tickets[b], 1u);
  if (old != (unsigned int)P.K) return;
  __threadfence();
  int nacc = P.K, bad = 0;
  const volatile unsigned long long* u = P.ws_units + (size_t)b * (P.K + 1);
  for (int q = 0; q <= P.K; ++q) {
    const unsigned long long rec = u[q];
    bad |= (int)((rec >> 33) & 1ull);
    if (q < P.K && nacc == P.K && !((rec >> 32) & 1ull)) nacc = q;
  }
  const int last = (int)(uint32_t)u[nacc];
  int32_t* ot = P.out_tokens + (size_t)b * (P.K + 1);
  for (int q = 0; q <= P.K; ++q) {
    int v = -1;
    if (!bad) v = q < nacc ? P.dtok[(size_t)b * P.K + q] : (q == nacc ? last : -1);
    ot[q] = v;
  }
  P.out_n[b] = bad ? -1 : nacc;
  for (int q = 0; q <= P.K; ++q) P.ws_units[(size_t)b * (P.K + 1) + q] = 0ull;
  P.ws_tickets[b] = 0u;
}

// ------------------------------------------------------------------------
// Exact cut over n gathered entries (composite (key << 32) | ~id, n <= GCAP),
// run by the whole CTA. Sorting the composites in descending order gives the
// token order (logit desc, id asc). Top-k rows: the first kk entries, then the
// top-p prefix inside them. Top-p rows: entries after `above` mass, cut where
// the exclusive mass reaches X. Writes thr/tie/ZL (kept iff key > thr or key
// == thr and id <= tie).
__device__ void local_select(unsigned long long* g, int n, const RowK& rk, float fscale,
                             uint32_t kmask, unsigned long long* scan, uint32_t* out_thr,
                             int* out_tie, unsigned long long* out_zl, int* out_fail) {
  const int tid = threadIdx.x;
  int N = 2;
  while (N < n) N <<= 1;
  for (int p = n + tid; p < N; p += NT) g[p] = 0ull;
  __syncthreads();
  for (int k = 2; k <= N; k <<= 1) {              // bitonic sort, descending
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int p = tid; p < N; p += NT) {
        const int q = p ^ j;
        if (q > p) {
          const unsigned long long a = g[p], c = g[q];
          const bool desc = (p & k) == 0;
          if (desc ? (a < c) : (a > c)) {
            g[p] = c;
            g[q] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  constexpr int PER = GCAP / NT;
  unsigned long long e[PER];
  unsigned long long s = 0;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int p = tid * PER + u;
    e[u] = 0;
    if (p < n) {
      const uint32_t key = (uint32_t)(g[p] >> 32);
      e[u] = to_fixed(hweight(mkey_to_float(key, kmask), rk.w), fscale);
    }
    s += e[u];
  }
  unsigned long long tot;
  const unsigned long long base = block_excl_scan<unsigned long long>(s, scan, &tot);
  int limit = n;
  double X = rk.X;
  unsigned long long above = rk.above;
  const bool topp = rk.topp < 1.0f;
  __shared__ unsigned long long z1s;
  __shared__ unsigned int kept_s;
  if (rk.mode == RM_TOPK) {
    limit = min(n, rk.kk);
    above = 0;
    if (tid == 0) z1s = 0;
    __syncthreads();
    unsigned long long run = base;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int p = tid * PER + u;
      if (p == limit - 1) z1s = run + e[u];
      run += e[u];
    }
    __syncthreads();
    X = (double)rk.topp * (double)z1s;
  }
  unsigned int c = 0;
  {
    unsigned long long run = base;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int p = tid * PER + u;
      if (p < limit && (!topp || (double)(above + run) < X)) ++c;
      run += e[u];
    }
  }
  unsigned int kept = block_sum<unsigned int>(c, (unsigned int*)scan);
  if (rk.mode == RM_TOPK && kept < 1) kept = 1;
  if (tid == 0) kept_s = kept;
  __syncthreads();
  kept = kept_s;
  if (tid == 0) {
    if (kept == 0) {
      // the cut lies just above the listed range: keep only what is above it
      *out_thr = (uint32_t)(g[0] >> 32);
      *out_tie = -1;
      *out_zl = above;
    } else {
      const unsigned long long last = g[kept - 1];
      *out_thr = (uint32_t)(last >> 32);
      *out_tie = (int)(~(uint32_t)last);
    }
    *out_fail = (rk.mode == RM_TOPK && n < rk.kk) ? 1 : 0;
  }
  {
    unsigned long long run = base;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int p = tid * PER + u;
      if (kept > 0 && p == (int)kept - 1) *out_zl = above + run + e[u];
      run += e[u];
    }
  }
  __syncthreads();
}

// Logit j of a row slice in shared memory (plain loads the compiler schedules).
template <typename DT>
__device__ __forceinline__ float ld_logit(const unsigned char* base, int j) {
  return to_f32<DT>(reinterpret_cast<const DT*>(base)[j]);
}
// Two consecutive logits j, j+1 (j even) of a bf16 row from one 32-bit word.
__device__ __forceinline__ void ld_pair(const unsigned char* base, int j, float& z0, float& z1) {
  const uint32_t w = reinterpret_cast<const uint32_t*>(base)[j >> 1];
  z0 = __uint_as_float(w << 16);
  z1 = __uint_as_float(w & 0xffff0000u);
}

// Pass B over one row slice: see the file header. zh: fixed-point head mass,
// zt: fp32 tail mass (full-support rows), histograms in pm/pc (stride NT).
template <typename DT>
__device__ __forceinline__ void passB_row(const unsigned char* base, int j0, int j1, int ept,
                                          int mode, const RowW w, uint32_t tau, uint32_t kmask,
                                          float fscale, float* pm, uint8_t* pc, uint16_t* list,
                                          unsigned int* lcnt, unsigned long long& zh, float& zt) {
  constexpr int PAIR = sizeof(DT) == 2 ? 2 : 1;
  auto topp_elem = [&](float z) -> bool {
    const float e = hweight(z, w);
    if (z >= w.zh) {
      zh += to_fixed(e, fscale);
      return true;
    }
    const float dd = tail_dist(z, w);
    const int bb = dd < 16.0f ? (int)dd : NB;
    pm[bb * NT] += e;
    pc[bb * NT] += 1;
    return false;
  };
  for (int s = 0; s < ept; s += PAIR) {
    const int j = j0 + s;
    float z[2];
    bool v[2];
    if (PAIR == 2) {
      v[0] = j < j1;
      v[1] = j + 1 < j1;
      if (v[0]) ld_pair(base, j, z[0], z[1]);
    } else {
      v[0] = j < j1;
      if (v[0]) z[0] = ld_logit<DT>(base, j);
    }
#pragma unroll
    for (int k = 0; k < PAIR; ++k) {
      bool in = false;
      if (v[k]) {
        if (mode == RM_TOPK) {
          in = mkey(z[k], kmask) >= tau;
        } else if (mode == RM_TOPP) {
          in = topp_elem(z[k]);
        } else {
          const float e = hweight(z[k], w);
          if (z[k] >= w.zh) zh += to_fixed(e, fscale);
          else zt += e;
        }
      }
      if (mode != RM_FULL) list_push(in, (uint16_t)(j + k), list, lcnt, LCAP);
    }
  }
}

// One refinement pass over the tail tokens of range q at level lev - 1:
// mass/count per sub-bin of level lev, and the key range of those tokens.
template <typename DT>
__device__ __forceinline__ void refine_row(const unsigned char* base, int j0, int j1, const RowW w,
                                           int q, float sc_prev, float sc_cur, uint32_t kmask,
                                           float* pm, uint8_t* pc, uint32_t& kmn, uint32_t& kmx) {
  for (int j = j0; j < j1; ++j) {
    const float z = ld_logit<DT>(base, j);
    if (z >= w.zh) continue;
    const float dd = tail_dist(z, w);
    if (dd >= 16.0f || (int)(dd * sc_prev) != q) continue;
    const int sub = ((int)(dd * sc_cur)) & (NB - 1);
    pm[sub * NT] += hweight(z, w);
    pc[sub * NT] += 1;
    const uint32_t key = mkey(z, kmask);
    kmn = min(kmn, key);
    kmx = max(kmx, key);
  }
}

// Lists the tail tokens of range q at level lev (scale = 16^lev).
template <typename DT>
__device__ __forceinline__ void list_range_row(const unsigned char* base, int j0, int j1, int ept,
                                               const RowW w, int q, float scl, uint16_t* list,
                                               unsigned int* lcnt) {
  for (int s = 0; s < ept; ++s) {
    const int j = j0 + s;
    bool in = false;
    if (j < j1) {
      const float z = ld_logit<DT>(base, j);
      if (z < w.zh) {
        const float dd = tail_dist(z, w);
        in = dd < 16.0f && (int)(dd * scl) == q;
      }
    }
    list_push(in, (uint16_t)j, list, lcnt, LCAP);
  }
}

// Token id of the target-th (0-based) member, in id order, of the tie group
// {key == thr} of each row flagged in `want`; NO_TIE for rows not flagged.
// Every CTA of the cluster calls it (two cluster barriers). Per-thread ranges
// are contiguous and CTAs hold consecutive slices, so thread order and CTA
// order are token-id order.
template <typename DT>
__device__ void tie_split(const bool want[2], const uint32_t thr[2], const unsigned int target[2],
                          const unsigned char* rb0, const unsigned char* rb1, int j0, int j1,
                          int v0, uint32_t kmask, Work& W, int& xb, uint32_t C, uint32_t rank,
                          int out[2]) {
  const int tid = threadIdx.x;
  unsigned int cnt[2] = {0, 0};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (!want[r]) continue;
    const unsigned char* rb = r == 0 ? rb0 : rb1;
    for (int j = j0; j < j1; ++j) cnt[r] += (mkey(ld_logit<DT>(rb, j), kmask) == thr[r]);
  }
  unsigned int excl[2], tot[2];
  excl[0] = block_excl_scan<unsigned int>(cnt[0], W.scan32, &tot[0]);
  excl[1] = block_excl_scan<unsigned int>(cnt[1], W.scan32, &tot[1]);
  const int buf = xb;
  xb ^= 1;
  if (tid == 0) {
    W.xs[buf][0] = tot[0];
    W.xs[buf][1] = tot[1];
  }
  __syncthreads();
  cluster_sync();
  int found[2] = {NO_TIE, NO_TIE};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (!want[r]) continue;
    unsigned int off = 0;
    for (uint32_t q = 0; q < rank; ++q) off += (unsigned int)ld_peer_u64(&W.xs[buf][r], q);
    const unsigned int lo = off + excl[r];
    if (cnt[r] > 0 && target[r] >= lo && target[r] < lo + cnt[r]) {
      const unsigned char* rb = r == 0 ? rb0 : rb1;
      unsigned int seen = lo;
      for (int j = j0; j < j1; ++j)
        if (mkey(ld_logit<DT>(rb, j), kmask) == thr[r]) {
          if (seen == target[r]) {
            found[r] = v0 + j;
            break;
          }
          ++seen;
        }
    }
  }
  const int buf2 = xb;
  xb ^= 1;
  if (tid < 2) W.xs[buf2][tid] = NO_TIE;
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 2; ++r)
    if (found[r] != NO_TIE) W.xs[buf2][r] = (unsigned long long)found[r];
  __syncthreads();
  cluster_sync();
  if (tid < 2) {
    int f = NO_TIE;
    for (uint32_t q = 0; q < C; ++q) f = min(f, (int)ld_peer_u64(&W.xs[buf2][tid], q));
    W.bi[6 + tid] = f;
  }
  __syncthreads();
  out[0] = W.bi[6];
  out[1] = W.bi[7];
  __syncthreads();
}

// ------------------------------------------------------------------------
template <typename DT, int MODE>
__global__ void __launch_bounds__(NT, 3) sv_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t C = cluster_size();
  const uint32_t rank = cluster_rank();
  const int unit = blockIdx.x / C;
  const int tid = threadIdx.x;
  const int V = P.V;
  const int es = (int)sizeof(DT);
  const size_t row_bytes = ((size_t)P.slice * es + 15) & ~(size_t)15;
  Work& W = *reinterpret_cast<Work*>(smem + 2 * row_bytes);
  const uint32_t sb0 = smem_addr(smem);                 // shared addresses (DSMEM peers)
  const uint32_t sb1 = smem_addr(smem + row_bytes);
  const unsigned char* rb0 = smem;                       // row slices for local loads
  const unsigned char* rb1 = smem + row_bytes;
  const uint32_t kmask = P.keymask;
  const float fscale = P.fix_scale;

  // ---------------------------------------------------------------- unit
  int b, i, seq;
  const DT* g0;
  const DT* g1 = nullptr;
  if (MODE == MODE_VERIFY) {
    b = unit / (P.K + 1);
    i = unit % (P.K + 1);
    seq = b;
    g0 = reinterpret_cast<const DT*>(P.rows0) + ((size_t)b * (P.K + 1) + i) * V;
  } else if (MODE == MODE_SAMPLE) {
    b = unit / P.K;
    i = unit % P.K;
    seq = b;
    g0 = reinterpret_cast<const DT*>(P.rows0) + (size_t)unit * V;
  } else {
    b = unit;
    i = 0;
    seq = unit;
    g0 = reinterpret_cast<const DT*>(P.rows0) + (size_t)unit * V;
  }
  const float T = P.temp[seq];
  const int topk = P.topk[seq];
  const float topp = P.topp[seq];
  const bool greedy = (T == 0.0f);
  bool param_bad = !(T >= 0.0f) || !(topp > 0.0f) || topk < 0;   // NaN fails >= and >
  int dtok = -1;
  if (MODE == MODE_VERIFY && i < P.K) {
    dtok = P.dtok[(size_t)b * P.K + i];
    if (dtok < 0 || dtok >= V) param_bad = true;
  }
  int nrows = 1;
  if (MODE == MODE_VERIFY && i < P.K && !greedy && !param_bad) {
    if (P.rows1 == nullptr) {
      param_bad = true;
    } else {
      nrows = 2;
      g1 = reinterpret_cast<const DT*>(P.rows1) + ((size_t)b * P.K + i) * V;
    }
  }
  SV_MARK(0);
  const int v0 = (int)rank * P.slice;
  const int n = max(0, min(V, v0 + P.slice) - v0);

  // ---------------------------------------------------------------- load
  if (tid == 0) {
    mbar_init(&W.mbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  int load_bad = 0;
  if (P.bulk_ok) {
    if (tid == 0) {
      const uint32_t bytes = (uint32_t)(n * es);
      mbar_arrive_expect_tx(&W.mbar, bytes * nrows);
      const uint64_t pol = policy_evict_first();
      for (int r = 0; r < nrows; ++r) {
        const char* src = reinterpret_cast<const char*>((r == 0 ? g0 : g1) + v0);
        char* dst = reinterpret_cast<char*>(smem + (r == 0 ? 0 : row_bytes));
        for (uint32_t off = 0; off < bytes; off += 32768u) {
          const uint32_t sz = min(32768u, bytes - off);
          bulk_g2s(dst + off, src + off, sz, &W.mbar, pol);
        }
      }
    }
    if (!mbar_wait_bounded(&W.mbar, 0, WAIT_LIMIT_NS)) {
      load_bad = 1;
      if (tid == 0) atomicOr(P.ws_error, 1u);
    }
  } else {
    DT* d0 = reinterpret_cast<DT*>(smem);
    DT* d1 = reinterpret_cast<DT*>(smem + row_bytes);
    for (int j = tid; j < n; j += NT) d0[j] = g0[v0 + j];
    if (nrows == 2)
      for (int j = tid; j < n; j += NT) d1[j] = g1[v0 + j];
    __syncthreads();
  }
  SV_MARK(1);
  const int j0 = tid * P.ept;
  const int j1 = min(n, j0 + P.ept);
  const int ept = P.ept;

  // ------------------------------------------- pass A: max, argmax, NaN
  const bool topk_on = topk > 0 && topk < V;
  const int kk = topk_on ? topk : V;
  float best[2] = {-INFINITY, -INFINITY};
  int bidx[2] = {0x7fffffff, 0x7fffffff};
  int bad[2] = {0, 0};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r < nrows) {
      const unsigned char* rb = r == 0 ? rb0 : rb1;
      float bb = -INFINITY;
      int bi = 0x7fffffff, bd = 0;
      for (int j = j0; j < j1; ++j) {
        const float z = ld_logit<DT>(rb, j);
        bd |= !(z <= 3.402823466e38f);        // NaN or +inf
        if (z > bb) {
          bb = z;
          bi = j;
        }
      }
      best[r] = bb;
      bidx[r] = bi;
      bad[r] = bd;
    }
  }
  uint32_t kth[2] = {KEY_ALL, KEY_ALL};
  if (!greedy && topk_on && kk <= NT) {
#pragma unroll
    for (int r = 0; r < 2; ++r)
      if (r < nrows)
        kth[r] = block_kth_largest(mkey(best[r], kmask), j1 > j0, kk, W.kthh[r], W.scan32, P.nlev);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    for (int o = 16; o; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best[r], o);
      const int oi = __shfl_xor_sync(0xffffffffu, bidx[r], o);
      if (ob > best[r] || (ob == best[r] && oi < bidx[r])) {
        best[r] = ob;
        bidx[r] = oi;
      }
      bad[r] |= __shfl_xor_sync(0xffffffffu, bad[r], o);
    }
  }
  {
    __shared__ float sbest[2][NWARP];
    __shared__ int sidx[2][NWARP], sbad[2][NWARP];
    if (lane_id() == 0)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        sbest[r][warp_id()] = best[r];
        sidx[r][warp_id()] = bidx[r];
        sbad[r][warp_id()] = bad[r];
      }
    __syncthreads();
    if (tid < 2) {
      const int r = tid;
      float bb = -INFINITY;
      int ii = 0x7fffffff, bd = load_bad;
      for (int w = 0; w < NWARP; ++w) {
        if (sbest[r][w] > bb || (sbest[r][w] == bb && sidx[r][w] < ii)) {
          bb = sbest[r][w];
          ii = sidx[r][w];
        }
        bd |= sbad[r][w];
      }
      W.xa[r].best = bb;
      W.xa[r].best_id = (ii == 0x7fffffff) ? 0x7fffffff : v0 + ii;
      W.xa[r].bad = bd;
      W.xa[r].kth = r == 0 ? kth[0] : kth[1];
    }
  }
  __syncthreads();
  SV_MARK(2);
  cluster_sync();  // X1
  SV_MARK(3);
  if (tid < 2) {
    const int r = tid;
    float bb = -INFINITY;
    int ii = 0x7fffffff, bd = 0;
    uint32_t kt = KEY_ALL;
    for (uint32_t c = 0; c < C; ++c) {
      const float pb = ld_peer_f32(&W.xa[r].best, c);
      const int pi = (int)ld_peer_u32(&W.xa[r].best_id, c);
      if (pb > bb || (pb == bb && pi < ii)) {
        bb = pb;
        ii = pi;
      }
      bd |= (int)ld_peer_u32(&W.xa[r].bad, c);
      kt = max(kt, ld_peer_u32(&W.xa[r].kth, c));
    }
    RowK& rk = W.rk[r];
    rk.w.m = bb;
    rk.argmax = ii;
    rk.bad = bd | (bb == -INFINITY ? 1 : 0);
    rk.tau = kt;
    rk.kk = kk;
    rk.topp = topp;
    rk.thr = KEY_ALL;
    rk.tie = NO_TIE;
    rk.ZL = 0;
    rk.Z = 0;
    rk.Zh = 0;
    rk.above = 0;
    rk.X = 0.0;
    rk.lev = -1;
    rk.q = 0;
    rk.need = ND_DONE;
    if (!greedy && !(bd | (bb == -INFINITY))) {
      // per-row weight constants, once per CTA (double precision on one thread)
      const double inv = 1.0 / (double)T;
      const double c2 = 1.4426950408889634 * inv;
      rk.w.c2 = (float)c2;
      rk.w.c2_lo = (float)(c2 - (double)rk.w.c2);
      rk.w.invT = (float)inv;
      rk.w.zh = (float)((double)bb - (double)DHEAD * (double)T);
      rk.mode = topk_on ? ((kk <= NT) ? RM_TOPK : -1) : (topp < 1.0f ? RM_TOPP : RM_FULL);
    } else {
      rk.mode = RM_FULL;
    }
  }
  __syncthreads();
  int xb = 0;            // next exchange buffer
  const bool unit_err = param_bad || W.rk[0].bad || (nrows == 2 && W.rk[1].bad);

  // --------------------------------------------------------- greedy / error
  if (greedy || unit_err) {
    const int am = W.rk[0].argmax;
    if (MODE == MODE_SAMPLE && rank == 0 && tid == 0) P.out_tokens[unit] = unit_err ? -1 : am;
    if (MODE == MODE_PROBS) {
      float* out = P.out_probs + (size_t)unit * V + v0;
      for (int j = tid; j < n; j += NT)
        out[j] = unit_err ? __int_as_float(0x7fc00000) : ((v0 + j == am) ? 1.0f : 0.0f);
    }
    cluster_sync();  // peers may still read this CTA's exchange slots
    if (MODE == MODE_VERIFY && rank == 0 && tid == 0)
      publish_unit(P, unit, b, unit_err ? -1 : am, !unit_err && i < P.K && dtok == am, unit_err);
    if (load_bad) mbar_wait_bounded(&W.mbar, 0, WAIT_LIMIT_NS);
    return;
  }

  // ------------------------------------------------------- pass B
  const RowW rw0 = W.rk[0].w, rw1 = W.rk[1].w;
  const int mode0 = W.rk[0].mode, mode1 = W.rk[1].mode;
  const uint32_t tau0 = W.rk[0].tau, tau1 = W.rk[1].tau;
  const bool general_k = (mode0 < 0);      // top-k with k beyond the per-thread pool
  if (tid < 2) W.lcnt[tid] = 0;
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r >= nrows || general_k) continue;
    const int mode = r == 0 ? mode0 : mode1;
    unsigned long long zh = 0;
    float zt = 0.f;
    if (mode == RM_TOPP) {
#pragma unroll
      for (int bb = 0; bb < NBH; ++bb) {
        W.u.ph.pmass[bb][tid] = 0.f;
        W.u.ph.pcnt[bb][tid] = 0;
      }
    }
    passB_row<DT>(r == 0 ? rb0 : rb1, j0, j1, ept, mode, r == 0 ? rw0 : rw1, r == 0 ? tau0 : tau1,
                  kmask, fscale, &W.u.ph.pmass[0][tid], &W.u.ph.pcnt[0][tid], W.list[r],
                  &W.lcnt[r], zh, zt);
    __syncthreads();
    XB& x = W.xb[xb][r];
    const unsigned long long zhs = block_sum<unsigned long long>(zh, W.scan64);
    const unsigned long long zts = block_sum<unsigned long long>(to_fixed(zt, fscale), W.scan64);
    if (mode == RM_TOPP) {
      // reduce the private histograms: warp w handles bins w, w + NWARP, ...
      for (int bb = warp_id(); bb < NBH; bb += NWARP) {
        unsigned long long m = 0;
        unsigned int c = 0;
        for (int t = lane_id(); t < NT; t += 32) {
          m += to_fixed(W.u.ph.pmass[bb][t], fscale);
          c += W.u.ph.pcnt[bb][t];
        }
        m = warp_sum(m);
        c = warp_sum(c);
        if (lane_id() == 0) {
          x.hm[bb] = m;
          x.hc[bb] = c;
        }
      }
    }
    if (tid == 0) {
      x.zh = zhs;
      x.zt = zts;
      x.lcnt = W.lcnt[r];
    }
    __syncthreads();
  }
  SV_MARK(4);
  cluster_sync();   // X2
  SV_MARK(5);
  // cluster totals and the next step of every row (thread r decides row r)
  if (tid < nrows && !general_k) {
    const int r = tid;
    RowK& rk = W.rk[r];
    unsigned long long zh = 0, zt = 0, hm[NBH];
    unsigned int hc[NBH], lc = 0, lmax = 0;
    for (int bb = 0; bb < NBH; ++bb) {
      hm[bb] = 0;
      hc[bb] = 0;
    }
    const XB* px = &W.xb[xb][r];
    for (uint32_t c = 0; c < C; ++c) {
      zh += ld_peer_u64(&px->zh, c);
      zt += ld_peer_u64(&px->zt, c);
      const unsigned int l = ld_peer_u32(&px->lcnt, c);
      rk.rc[c] = l;
      lc += l;
      lmax = max(lmax, l);
      if (rk.mode == RM_TOPP)
        for (int bb = 0; bb < NBH; ++bb) {
          hm[bb] += ld_peer_u64(&px->hm[bb], c);
          hc[bb] += ld_peer_u32(&px->hc[bb], c);
        }
    }
    rk.Zh = zh;
    if (rk.mode == RM_FULL) {
      rk.Z = zh + zt;
      rk.ZL = rk.Z;
      rk.need = ND_DONE;
    } else if (rk.mode == RM_TOPK) {
      rk.need = (lc > GCAP || lmax > LCAP || lc < (unsigned int)rk.kk) ? ND_GENERAL : ND_LIST;
      rk.lev = -1;
    } else {
      unsigned long long z = zh;
      for (int bb = 0; bb < NBH; ++bb) z += hm[bb];
      rk.Z = z;
      rk.X = (double)rk.topp * (double)z;
      if ((double)zh >= rk.X) {            // the cut lies in the head
        rk.lev = -1;
        rk.above = 0;
        rk.need = (lc > GCAP || lmax > LCAP) ? ND_GENERAL : ND_LIST;
      } else {
        // first bin (by distance) where the cumulative mass reaches X; the
        // last non-empty bin if rounding keeps the total just below X
        unsigned long long cum = zh, pick_above = zh;
        int pick = -1;
        for (int bb = 0; bb < NBH; ++bb) {
          if (hc[bb] == 0) continue;
          pick = bb;
          pick_above = cum;
          if ((double)(cum + hm[bb]) >= rk.X) break;
          cum += hm[bb];
        }
        if (pick < 0 || pick == NB) {
          rk.need = ND_GENERAL;
        } else {
          rk.lev = 0;
          rk.q = pick;
          rk.above = pick_above;
          unsigned int cmax = 0;
          for (uint32_t c = 0; c < C; ++c) {
            const unsigned int cc = ld_peer_u32(&px->hc[pick], c);
            rk.rc[c] = cc;
            cmax = max(cmax, cc);
          }
          rk.need = (hc[pick] <= GCAP && cmax <= LCAP) ? ND_LIST : ND_REFINE;
        }
      }
    }
  }
  xb ^= 1;
  __syncthreads();
#ifdef SV_TRACE
  if (tid == 0 && rank == 0 && unit < 256)
    g_trace[unit * 16 + 13] = (unsigned long long)W.rk[1].need | ((unsigned long long)(W.rk[1].lev + 1) << 8) |
                              ((unsigned long long)W.rk[1].q << 16) | ((unsigned long long)W.rk[1].rc[0] << 32);
#endif

  // ------------------------------------------------- refinement of top-p cuts
  for (int lev = 1; lev <= MAXLEV && !general_k; ++lev) {
    bool any = false;
#pragma unroll
    for (int r = 0; r < 2; ++r)
      if (r < nrows && W.rk[r].need == ND_REFINE) any = true;
    if (!any) break;
    const float sc_prev = pow16(lev - 1), sc_cur = pow16(lev);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r >= nrows || W.rk[r].need != ND_REFINE) continue;
      const int q = W.rk[r].q;
#pragma unroll
      for (int bb = 0; bb < NB; ++bb) {
        W.u.ph.pmass[bb][tid] = 0.f;
        W.u.ph.pcnt[bb][tid] = 0;
      }
      uint32_t kmn = 0xffffffffu, kmx = 0u;
      refine_row<DT>(r == 0 ? rb0 : rb1, j0, j1, r == 0 ? rw0 : rw1, q, sc_prev, sc_cur, kmask,
                     &W.u.ph.pmass[0][tid], &W.u.ph.pcnt[0][tid], kmn, kmx);
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        kmn = min(kmn, __shfl_xor_sync(0xffffffffu, kmn, o));
        kmx = max(kmx, __shfl_xor_sync(0xffffffffu, kmx, o));
      }
      if (lane_id() == 0) {                   // kthh is free after pass A: key-range scratch
        W.kthh[0][warp_id()] = kmn;
        W.kthh[1][warp_id()] = kmx;
      }
      __syncthreads();
      XB& x = W.xb[xb][r];
      if (tid == 0) {
        uint32_t a = 0xffffffffu, bmax = 0u;
        for (int w = 0; w < NWARP; ++w) {
          a = min(a, W.kthh[0][w]);
          bmax = max(bmax, W.kthh[1][w]);
        }
        x.kmin = a;
        x.kmax = bmax;
      }
      for (int bb = warp_id(); bb < NB; bb += NWARP) {
        unsigned long long m = 0;
        unsigned int c = 0;
        for (int t = lane_id(); t < NT; t += 32) {
          m += to_fixed(W.u.ph.pmass[bb][t], fscale);
          c += W.u.ph.pcnt[bb][t];
        }
        m = warp_sum(m);
        c = warp_sum(c);
        if (lane_id() == 0) {
          x.hm[bb] = m;
          x.hc[bb] = c;
        }
      }
      __syncthreads();
    }
    cluster_sync();   // X3..
    if (tid < nrows && W.rk[tid].need == ND_REFINE) {
      const int r = tid;
      RowK& rk = W.rk[r];
      unsigned long long hm[NB];
      unsigned int hc[NB];
      for (int bb = 0; bb < NB; ++bb) {
        hm[bb] = 0;
        hc[bb] = 0;
      }
      const XB* px = &W.xb[xb][r];
      uint32_t kmn = 0xffffffffu, kmx = 0u;
      for (uint32_t c = 0; c < C; ++c) {
        for (int bb = 0; bb < NB; ++bb) {
          hm[bb] += ld_peer_u64(&px->hm[bb], c);
          hc[bb] += ld_peer_u32(&px->hc[bb], c);
        }
        kmn = min(kmn, ld_peer_u32(&px->kmin, c));
        kmx = max(kmx, ld_peer_u32(&px->kmax, c));
      }
      if (kmn == kmx) {
        // the range holds one logit value: keep the first j members (by id)
        // whose exclusive mass stays below X
        unsigned int cnt = 0;
        for (int bb = 0; bb < NB; ++bb) cnt += hc[bb];
        const unsigned long long Et = to_fixed(hweight(mkey_to_float(kmn, kmask), rk.w), fscale);
        double jf = Et > 0 ? ceil((rk.X - (double)rk.above) / (double)Et) : (double)cnt;
        jf = fmin(fmax(jf, 0.0), (double)cnt);
        const unsigned int j = (unsigned int)jf;
        rk.thr = kmn;
        rk.jt = j;
        rk.ZL = rk.above + (unsigned long long)j * Et;
        rk.tie = j == 0 ? -1 : NO_TIE;
        rk.need = (j == 0 || j == cnt) ? ND_DONE : ND_TIE;
      } else {
        unsigned long long cum = rk.above, pick_above = rk.above;
        int pick = -1;
        for (int bb = 0; bb < NB; ++bb) {
          if (hc[bb] == 0) continue;
          pick = bb;
          pick_above = cum;
          if ((double)(cum + hm[bb]) >= rk.X) break;
          cum += hm[bb];
        }
        if (pick < 0) {
          rk.need = ND_GENERAL;
        } else {
          rk.lev = lev;
          rk.q = rk.q * NB + pick;
          rk.above = pick_above;
          unsigned int cmax = 0;
          for (uint32_t c = 0; c < C; ++c) {
            const unsigned int cc = ld_peer_u32(&px->hc[pick], c);
            rk.rc[c] = cc;
            cmax = max(cmax, cc);
          }
          if (hc[pick] <= GCAP && cmax <= LCAP) rk.need = ND_LIST;
          else if (lev == MAXLEV) rk.need = ND_GENERAL;
        }
      }
    }
    xb ^= 1;
    __syncthreads();
  }

  // ------------------------------------- single-value ranges: split by id
  {
    bool want[2] = {false, false};
    uint32_t tthr[2] = {0, 0};
    unsigned int tgt[2] = {0, 0};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      want[r] = r < nrows && W.rk[r].need == ND_TIE;
      tthr[r] = W.rk[r].thr;
      tgt[r] = W.rk[r].jt - 1;
    }
    if (want[0] || want[1]) {
      int found[2];
      tie_split<DT>(want, tthr, tgt, rb0, rb1, j0, j1, v0, kmask, W, xb, C, rank, found);
      if (tid < 2 && want[tid]) {
        W.rk[tid].tie = found[tid];
        W.rk[tid].need = ND_DONE;
      }
      __syncthreads();
    }
  }

  // ---------------------------------------------- lists -> selecting CTA
  bool general = general_k;
#pragma unroll
  for (int r = 0; r < 2; ++r)
    if (r < nrows && (W.rk[r].need == ND_GENERAL || W.rk[r].need == ND_REFINE)) general = true;
  if (!general) {
    // list the range of rows whose cut lies in a tail range
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r >= nrows || W.rk[r].need != ND_LIST || W.rk[r].lev < 0) continue;
      if (tid == 0) W.lcnt[r] = 0;
      __syncthreads();
      list_range_row<DT>(r == 0 ? rb0 : rb1, j0, j1, ept, r == 0 ? rw0 : rw1, W.rk[r].q,
                         pow16(W.rk[r].lev), W.list[r], &W.lcnt[r]);
    }
    __syncthreads();
    // push the entries into CTA 0's gather buffer (the union is free there:
    // CTA 0 finished its histograms before the last cluster barrier)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r >= nrows || W.rk[r].need != ND_LIST) continue;
      unsigned int off = 0;
      for (uint32_t c = 0; c < rank; ++c) off += W.rk[r].rc[c];
      const unsigned int cnt = min(W.rk[r].rc[rank], (unsigned int)LCAP);
      const unsigned char* rb = r == 0 ? rb0 : rb1;
      for (unsigned int t = tid; t < cnt; t += NT) {
        const int j = W.list[r][t];
        const uint32_t key = mkey(ld_logit<DT>(rb, j), kmask);
        const uint32_t id = (uint32_t)(v0 + j);
        st_peer_u64(&W.u.g[r][off + t], 0, ((unsigned long long)key << 32) | (unsigned long long)(~id));
      }
    }
    cluster_sync();   // entries in place
    if (rank == 0) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (r >= nrows || W.rk[r].need != ND_LIST) continue;
        unsigned int tot = 0;
        for (uint32_t c = 0; c < C; ++c) tot += W.rk[r].rc[c];
        local_select(W.u.g[r], (int)tot, W.rk[r], fscale, kmask, W.scan64, &W.res_thr[r],
                     &W.res_tie[r], &W.res_zl[r], &W.res_fail[r]);
      }
    }
    cluster_sync();   // results in place at CTA 0
    if (tid < nrows && W.rk[tid].need == ND_LIST) {
      const int r = tid;
      RowK& rk = W.rk[r];
      rk.thr = ld_peer_u32(&W.res_thr[r], 0);
      rk.tie = (int)ld_peer_u32(&W.res_tie[r], 0);
      rk.ZL = ld_peer_u64(&W.res_zl[r], 0);
      rk.need = ld_peer_u32(&W.res_fail[r], 0) ? ND_GENERAL : ND_DONE;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 2; ++r)
      if (r < nrows && W.rk[r].need == ND_GENERAL) general = true;
  }
  SV_MARK(6);
#ifdef SV_TRACE
  if (tid == 0 && rank == 0 && unit < 256) {
    g_trace[unit * 16 + 10] = (unsigned long long)W.rk[0].need | ((unsigned long long)(W.rk[0].lev + 1) << 8) |
                              ((unsigned long long)W.rk[0].q << 16);
    g_trace[unit * 16 + 11] = (unsigned long long)W.rk[1].need | ((unsigned long long)(W.rk[1].lev + 1) << 8) |
                              ((unsigned long long)W.rk[1].q << 16);
    g_trace[unit * 16 + 12] = (unsigned long long)W.rk[1].mode | ((unsigned long long)W.rk[0].mode << 8);
  }
#endif

  // ------------------------------------------------- general selection path
  if (general) {
    const bool topp_on = topp < 1.0f;
    const bool any_sel = topk_on || topp_on;
    uint32_t gtau[2] = {KEY_ALL, KEY_ALL};
    if (topk_on) {
      if (kk <= NT) {
        gtau[0] = W.rk[0].tau;
        gtau[1] = W.rk[1].tau;
      }
    } else if (topp_on) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        // eligibility: within ln(V/(1-top_p)) + 0.05 nats of the maximum
        const float taud = logf((float)V / (1.0f - topp)) + 0.05f;
        const float zt = (r == 0 ? rw0.m : rw1.m) - taud * T;
        gtau[r] = isfinite(zt) ? mkey(zt, kmask) : KEY_ALL;
      }
    }
    uint32_t tk[2] = {0, 0};
    unsigned int jk[2] = {0, 0};
    unsigned long long Etk[2] = {0, 0};
    double Z1[2] = {0, 0};
    uint32_t thr[2] = {KEY_ALL, KEY_ALL};
    unsigned int jt[2] = {0, 0}, neq_all[2] = {0, 0};
    unsigned long long ZL[2] = {0, 0};
    for (int stage = 0; stage < 2 && any_sel; ++stage) {
      const bool by_mass = (stage == 1);
      if (stage == 0 && !topk_on) continue;
      if (stage == 1 && !topp_on) continue;
      uint32_t prefix[2] = {0, 0}, pmask = 0;
      unsigned int cabove[2] = {0, 0};
      unsigned long long mabove[2] = {0, 0};
      double need_m[2] = {0, 0};
      unsigned int lastcnt[2] = {0, 0};
      for (int lev = 0; lev < P.nlev; ++lev) {
        const int shift = 24 - 8 * lev;
        const int buf = xb;
        xb ^= 1;
        for (int t = tid; t < 2 * 256; t += NT) {
          W.u.gp.hcnt[buf][t >> 8][t & 255] = 0;
          W.u.gp.hmass[buf][t >> 8][t & 255] = 0;
        }
        __syncthreads();
        float zfar[2] = {0.f, 0.f};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (r >= nrows) continue;
          const unsigned char* rb = r == 0 ? rb0 : rb1;
          const RowW w = r == 0 ? rw0 : rw1;
          for (int j = j0; j < j1; ++j) {
            const float z = ld_logit<DT>(rb, j);
            const uint32_t key = mkey(z, kmask);
            bool in;
            if (stage == 0) {
              in = key >= gtau[r];
            } else if (topk_on) {
              in = key > tk[r];                   // the tie group at tk enters as one pseudo token
            } else {
              in = key >= gtau[r];
              if (!in && lev == 0) zfar[r] += hweight(z, w);
            }
            if (in && (key & pmask) == prefix[r]) {
              const unsigned int dg = (key >> shift) & 255u;
              atomicAdd(&W.u.gp.hcnt[buf][r][dg], 1u);
              const unsigned long long E = to_fixed(hweight(z, w), fscale);
              if (E) atomicAdd(&W.u.gp.hmass[buf][r][dg], E);
            }
          }
        }
        if (stage == 1 && topk_on && rank == 0 && tid == 0) {
#pragma unroll
          for (int r = 0; r < 2; ++r)
            if (r < nrows && (tk[r] & pmask) == prefix[r]) {
              const unsigned int dg = (tk[r] >> shift) & 255u;
              atomicAdd(&W.u.gp.hcnt[buf][r][dg], jk[r]);
              atomicAdd(&W.u.gp.hmass[buf][r][dg], (unsigned long long)jk[r] * Etk[r]);
            }
        }
        if (stage == 1 && !topk_on && lev == 0) {
          const unsigned long long zf0 = block_sum<unsigned long long>(to_fixed(zfar[0], fscale), W.scan64);
          const unsigned long long zf1 = block_sum<unsigned long long>(to_fixed(zfar[1], fscale), W.scan64);
          if (tid == 0) {
            W.xs[buf][0] = zf0;
            W.xs[buf][1] = zf1;
          }
        }
        __syncthreads();
        cluster_sync();
        for (int t = tid; t < 2 * 256; t += NT) {
          const int r = t >> 8, dg = t & 255;
          if (r < nrows) {
            unsigned int c = 0;
            unsigned long long w = 0;
            for (uint32_t q = 0; q < C; ++q) {
              c += ld_peer_u32(&W.u.gp.hcnt[buf][r][dg], q);
              w += ld_peer_u64(&W.u.gp.hmass[buf][r][dg], q);
            }
            W.u.gp.gcnt[r][dg] = c;
            W.u.gp.gmass[r][dg] = w;
          }
        }
        if (stage == 1 && !topk_on && lev == 0 && tid < nrows) {
          unsigned long long zf = 0;
          for (uint32_t q = 0; q < C; ++q) zf += ld_peer_u64(&W.xs[buf][tid], q);
          W.bu[2 + tid] = zf;
        }
        __syncthreads();
        if (stage == 1 && lev == 0) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            if (r >= nrows) continue;
            if (!topk_on) {
              unsigned long long s = 0;
              for (int dg = 0; dg < 256; ++dg) s += W.u.gp.gmass[r][dg];
              Z1[r] = (double)(s + W.bu[2 + r]);
            }
            need_m[r] = (double)topp * Z1[r];
          }
        }
        if (warp_id() < nrows) {
          const int r = warp_id();
          const unsigned int need_c =
              stage == 0 ? (unsigned int)kk - (r == 0 ? cabove[0] : cabove[1]) : 0u;
          const double need_mr =
              r == 0 ? need_m[0] - (double)mabove[0] : need_m[1] - (double)mabove[1];
          const DigitPick pk =
              pick_digit(W.u.gp.gcnt[r], W.u.gp.gmass[r], by_mass, need_c, need_mr);
          if (lane_id() == 0) {
            W.bi[r] = pk.digit;
            W.bi[2 + r] = (int)pk.cnt_above;
            W.bu[r] = pk.mass_above;
            W.bi[4 + r] = (int)W.u.gp.gcnt[r][pk.digit];
          }
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (r >= nrows) continue;
          prefix[r] |= (uint32_t)W.bi[r] << shift;
          cabove[r] += (unsigned int)W.bi[2 + r];
          mabove[r] += W.bu[r];
          lastcnt[r] = (unsigned int)W.bi[4 + r];
        }
        pmask |= 255u << shift;
        __syncthreads();
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (r >= nrows) continue;
        const unsigned long long Et =
            to_fixed(hweight(mkey_to_float(prefix[r], kmask), r == 0 ? rw0 : rw1), fscale);
        if (stage == 0) {
          tk[r] = prefix[r];
          jk[r] = (unsigned int)kk - cabove[r];
          Etk[r] = Et;
          Z1[r] = (double)(mabove[r] + (unsigned long long)jk[r] * Et);
          thr[r] = tk[r];
          jt[r] = jk[r];
          neq_all[r] = lastcnt[r];
          ZL[r] = mabove[r] + (unsigned long long)jk[r] * Et;
        } else {
          const double gap = need_m[r] - (double)mabove[r];
          const double jf = Et > 0 ? ceil(gap / (double)Et) : 1.0;
          const unsigned int j = (unsigned int)fmax(1.0, fmin(jf, (double)lastcnt[r]));
          thr[r] = prefix[r];
          jt[r] = j;
          neq_all[r] = (topk_on && prefix[r] == tk[r]) ? neq_all[r] : lastcnt[r];
          ZL[r] = mabove[r] + (unsigned long long)j * Et;
        }
      }
    }
    // tie split by token id
    bool need_tie[2] = {false, false};
#pragma unroll
    for (int r = 0; r < 2; ++r) need_tie[r] = r < nrows && any_sel && jt[r] < neq_all[r];
    int tie_res[2] = {NO_TIE, NO_TIE};
    if (need_tie[0] || need_tie[1]) {
      const unsigned int tgt[2] = {jt[0] - 1, jt[1] - 1};
      tie_split<DT>(need_tie, thr, tgt, rb0, rb1, j0, j1, v0, kmask, W, xb, C, rank, tie_res);
    }
    __syncthreads();
    if (tid < nrows) {
      const int r = tid;
      RowK& rk = W.rk[r];
      if (any_sel) {
        rk.thr = r == 0 ? thr[0] : thr[1];
        rk.ZL = r == 0 ? ZL[0] : ZL[1];
        rk.tie = (r == 0 ? need_tie[0] : need_tie[1]) ? (r == 0 ? tie_res[0] : tie_res[1]) : NO_TIE;
      } else {
        rk.thr = KEY_ALL;
        rk.tie = NO_TIE;
      }
    }
    __syncthreads();
  }
  SV_MARK(7);

  uint32_t thr[2];
  int tie[2];
  unsigned long long ZL[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    thr[r] = W.rk[r].thr;
    tie[r] = W.rk[r].tie;
    ZL[r] = W.rk[r].ZL;
  }
  auto kept = [&](int r, float z, int id) -> bool {
    const uint32_t key = mkey(z, kmask);
    const uint32_t t = r == 0 ? thr[0] : thr[1];
    const int ti = r == 0 ? tie[0] : tie[1];
    return key > t || (key == t && id <= ti);
  };

  // --------------------------------------------------- probabilities hook
  if (MODE == MODE_PROBS) {
    float* out = P.out_probs + (size_t)unit * V + v0;
    if (tid == 0) W.bu[0] = __double_as_longlong(1.0 / (double)ZL[0]);
    __syncthreads();
    const double inv = __longlong_as_double((long long)W.bu[0]);
    for (int j = tid; j < n; j += NT) {
      const float z = ld_logit<DT>(rb0, j);
      float pr = 0.0f;
      if (kept(0, z, v0 + j)) pr = (float)((double)to_fixed(hweight(z, rw0), fscale) * inv);
      out[j] = pr;
    }
    cluster_sync();
    return;
  }

  // ------------------------------------------------------------ acceptance
  bool flag = false;
  uint32_t ku, kv;
  philox_uniform_bits(P.seed, P.offset, (uint32_t)b, (uint32_t)i, &ku, &kv);
  const bool residual = (MODE == MODE_VERIFY && i < P.K);
  if (residual) {
    if (tid == 0) {
      const uint32_t owner = (uint32_t)(dtok / P.slice);
      const int jj = dtok - (int)owner * P.slice;
      double pq[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float z = ld_peer_logit<DT>(r == 0 ? sb0 : sb1, jj, owner);
        pq[r] = kept(r, z, dtok)
                    ? (double)to_fixed(hweight(z, r == 0 ? rw0 : rw1), fscale) /
                          (double)(r == 0 ? ZL[0] : ZL[1])
                    : 0.0;
      }
      W.bi[0] = ((double)ku * 5.9604644775390625e-08 * pq[1] < pq[0]) ? 1 : 0;
      W.bu[0] = __float_as_uint((float)((double)fscale / (double)ZL[0]));
      W.bu[1] = __float_as_uint((float)((double)fscale / (double)ZL[1]));
    }
    __syncthreads();
    flag = W.bi[0] != 0;
  }
  const float sp = residual ? __uint_as_float((uint32_t)W.bu[0]) : 0.f;
  const float sq = residual ? __uint_as_float((uint32_t)W.bu[1]) : 0.f;

  // ------------------------------------------- inverse-CDF in token-id order
  auto wgt = [&](int j, bool res) -> unsigned long long {
    const float z = ld_logit<DT>(rb0, j);
    if (!kept(0, z, v0 + j)) return 0ull;
    const float ep = hweight(z, rw0);
    if (!res) return to_fixed(ep, fscale);
    const float zq = ld_logit<DT>(rb1, j);
    // rounded products and difference (no FMA contraction): identical rows give d == 0
    const float q = kept(1, zq, v0 + j) ? __fmul_rn(hweight(zq, rw1), sq) : 0.0f;
    const float d = __fsub_rn(__fmul_rn(ep, sp), q);
    return d > 0.0f ? __float2ull_rz(d * 4611686018427387904.0f) : 0ull;
  };
  bool use_res = residual;
  for (int attempt = 0; attempt < 2; ++attempt) {
    unsigned long long s = 0;
    for (int j = j0; j < j1; ++j) s += wgt(j, use_res);
    unsigned long long ctot;
    const unsigned long long texcl = block_excl_scan<unsigned long long>(s, W.scan64, &ctot);
    const int buf = xb;
    xb ^= 1;
    if (tid == 0) W.xs[buf][0] = ctot;
    __syncthreads();
    cluster_sync();
    unsigned long long off = 0, S = 0;
    for (uint32_t q = 0; q < C; ++q) {
      const unsigned long long t = ld_peer_u64(&W.xs[buf][0], q);
      if (q < rank) off += t;
      S += t;
    }
    if (S == 0 && use_res) {       // (p - q)+ has no mass: sample from p
      use_res = false;
      continue;
    }
    const unsigned long long lo = off + texcl, hi = lo + s;
    const unsigned long long kvs = (unsigned long long)kv;
    if (s > 0 && !mul_gt(lo, 1ull << 24, kvs, S) && mul_gt(hi, 1ull << 24, kvs, S)) {
      unsigned long long run = lo;
      int tok = v0 + j1 - 1;
      for (int j = j0; j < j1; ++j) {
        run += wgt(j, use_res);
        if (mul_gt(run, 1ull << 24, kvs, S)) {
          tok = v0 + j;
          break;
        }
      }
      if (MODE == MODE_SAMPLE) P.out_tokens[unit] = tok;
      else publish_unit(P, unit, b, tok, flag, false);
    }
    break;
  }
  SV_MARK(8);
  cluster_sync();   // keep this CTA's shared memory alive until every peer is done
  SV_MARK(9);
}

__global__ void philox_kernel(uint64_t seed, uint64_t offset, int B, int K1, uint32_t* out) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= B * K1) return;
  uint32_t ku, kv;
  philox_uniform_bits(seed, offset, (uint32_t)(t / K1), (uint32_t)(t % K1), &ku, &kv);
  out[2 * t] = ku;
  out[2 * t + 1] = kv;
}

// ------------------------------------------------------------------ host
template <typename DT, int MODE>
cudaError_t launch(const Params& p, int C, size_t smem, cudaStream_t st) {
  auto kern = sv_kernel<DT, MODE>;
  static size_t configured = 0;      // largest dynamic shared memory set so far
  static bool nonportable = false;
  cudaError_t e;
  if (smem > configured) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  if (C > 8 && !nonportable) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    nonportable = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.nunits * C), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

struct Geometry {
  int C, slice, ept;
  size_t smem;
};

// Smallest cluster (1..16 CTAs) whose per-CTA share of two rows keeps the
// footprint near 72 KB (three CTAs per SM), else the largest that fits.
static Geometry geometry(int V, int es) {
  Geometry g{};
  const size_t target = 72 * 1024, hard = 227 * 1024;
  for (int C = 1; C <= 16; C *= 2) {
    int slice = (V + C - 1) / C;
    slice = (slice + 15) & ~15;
    const size_t rb = ((size_t)slice * es + 15) & ~(size_t)15;
    const size_t smem = 2 * rb + sizeof(Work);
    g.C = C;
    g.slice = slice;
    g.smem = smem;
    if (smem <= target) break;
    if (C == 16 && smem > hard) g.smem = 0;   // does not fit: reported as a shape error
  }
  // contiguous per-thread ranges with an odd number of 32-bit words (bank spread)
  int per = (g.slice + NT - 1) / NT;
  int words = (per * es + 3) / 4;
  words |= 1;
  g.ept = words * 4 / es;
  return g;
}

static int fix_scale_shift(int V) {
  int lg = 0;
  while ((1ll << lg) < (long long)V) ++lg;
  return 63 - lg;
}

}  // namespace sv

using namespace sv;

static sv_status check_common(int V, sv_dtype dt) {
  if (dt != SV_BF16 && dt != SV_F32) return SV_ERR_DTYPE;
  if (V < 2 || V > 262144) return SV_ERR_SHAPE;
  return SV_OK;
}

static bool fill_geometry(Params& p, int V, sv_dtype dt, Geometry* g) {
  const int es = dt == SV_BF16 ? 2 : 4;
  *g = geometry(V, es);
  p.V = V;
  p.slice = g->slice;
  p.ept = g->ept;
  p.nlev = dt == SV_BF16 ? 2 : 4;
  p.keymask = dt == SV_BF16 ? 0xFFFF0000u : 0xFFFFFFFFu;
  p.fix_scale = ldexpf(1.0f, fix_scale_shift(V));
  return g->smem != 0;
}

static sv_status do_launch(int mode, sv_dtype dt, const Params& p, const Geometry& g, cudaStream_t st) {
  cudaError_t e;
  if (dt == SV_BF16) {
    if (mode == MODE_VERIFY) e = launch<__nv_bfloat16, MODE_VERIFY>(p, g.C, g.smem, st);
    else if (mode == MODE_PROBS) e = launch<__nv_bfloat16, MODE_PROBS>(p, g.C, g.smem, st);
    else e = launch<__nv_bfloat16, MODE_SAMPLE>(p, g.C, g.smem, st);
  } else {
    if (mode == MODE_VERIFY) e = launch<float, MODE_VERIFY>(p, g.C, g.smem, st);
    else if (mode == MODE_PROBS) e = launch<float, MODE_PROBS>(p, g.C, g.smem, st);
    else e = launch<float, MODE_SAMPLE>(p, g.C, g.smem, st);
  }
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

static bool aligned(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

extern "C" {

size_t spec_verify_workspace_bytes(int B, int K) {
  if (B < 1 || K < 1) return 0;
  const size_t units = (size_t)B * (K + 1) * sizeof(unsigned long long);
  const size_t tickets = ((size_t)B * sizeof(unsigned int) + 15) & ~(size_t)15;
  return units + tickets + 16;
}

sv_status spec_verify(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      const int32_t* draft_tokens, const float* temperature, const int32_t* top_k,
                      const float* top_p, uint64_t philox_seed, uint64_t philox_offset, int B,
                      int K, int V, int32_t* out_tokens, int32_t* out_n_accepted, void* workspace,
                      size_t workspace_bytes, void* stream) {
  sv_status s = check_common(V, dtype);
  if (s != SV_OK) return s;
  if (B < 1 || B > 65535 || K < 1 || K > 16) return SV_ERR_SHAPE;
  if (!target_logits || !draft_tokens || !temperature || !top_k || !top_p || !out_tokens ||
      !out_n_accepted || !workspace)
    return SV_ERR_NULL;
  const size_t es = dtype == SV_BF16 ? 2 : 4;
  if (!aligned(target_logits, es) || (draft_logits && !aligned(draft_logits, es)) ||
      !aligned(draft_tokens, 4) || !aligned(temperature, 4) || !aligned(top_k, 4) ||
      !aligned(top_p, 4) || !aligned(out_tokens, 4) || !aligned(out_n_accepted, 4))
    return SV_ERR_ALIGN;
  if (!aligned(workspace, 16) || workspace_bytes < spec_verify_workspace_bytes(B, K))
    return SV_ERR_WORKSPACE;
  Params p{};
  Geometry g;
  if (!fill_geometry(p, V, dtype, &g)) return SV_ERR_SHAPE;
  p.rows0 = target_logits;
  p.rows1 = draft_logits;
  p.dtok = draft_tokens;
  p.temp = temperature;
  p.topk = top_k;
  p.topp = top_p;
  p.seed = philox_seed;
  p.offset = philox_offset;
  p.B = B;
  p.K = K;
  p.nunits = B * (K + 1);
  p.bulk_ok = ((V * es) % 16 == 0) && aligned(target_logits, 16) &&
              (!draft_logits || aligned(draft_logits, 16));
  p.out_tokens = out_tokens;
  p.out_n = out_n_accepted;
  char* ws = static_cast<char*>(workspace);
  p.ws_units = reinterpret_cast<unsigned long long*>(ws);
  p.ws_tickets = reinterpret_cast<unsigned int*>(ws + (size_t)p.nunits * 8);
  p.ws_error = reinterpret_cast<unsigned int*>(
      ws + (size_t)p.nunits * 8 + (((size_t)B * 4 + 15) & ~(size_t)15));
  return do_launch(MODE_VERIFY, dtype, p, g, static_cast<cudaStream_t>(stream));
}

sv_status spec_truncated_probs(const void* logits, sv_dtype dtype, int R, int V,
                               const float* temperature, const int32_t* top_k,
                               const float* top_p, float* out_probs, void* stream) {
  sv_status s = check_common(V, dtype);
  if (s != SV_OK) return s;
  if (R < 1 || R > (1 << 20)) return SV_ERR_SHAPE;
  if (!logits || !temperature || !top_k || !top_p || !out_probs) return SV_ERR_NULL;
  const size_t es = dtype == SV_BF16 ? 2 : 4;
  if (!aligned(logits, es) || !aligned(out_probs, 4)) return SV_ERR_ALIGN;
  Params p{};
  Geometry g;
  if (!fill_geometry(p, V, dtype, &g)) return SV_ERR_SHAPE;
  p.rows0 = logits;
  p.temp = temperature;
  p.topk = top_k;
  p.topp = top_p;
  p.B = R;
  p.K = 1;
  p.nunits = R;
  p.bulk_ok = ((V * es) % 16 == 0) && aligned(logits, 16);
  p.out_probs = out_probs;
  return do_launch(MODE_PROBS, dtype, p, g, static_cast<cudaStream_t>(stream));
}

sv_status spec_sample(const void* logits, sv_dtype dtype, int B, int K, int V,
                      const float* temperature, const int32_t* top_k, const float* top_p,
                      uint64_t philox_seed, uint64_t philox_offset, int32_t* out_tokens,
                      void* stream) {
  sv_status s = check_common(V, dtype);
  if (s != SV_OK) return s;
  if (B < 1 || B > 65535 || K < 1 || K > 16) return SV_ERR_SHAPE;
  if (!logits || !temperature || !top_k || !top_p || !out_tokens) return SV_ERR_NULL;
  const size_t es = dtype == SV_BF16 ? 2 : 4;
  if (!aligned(logits, es) || !aligned(out_tokens, 4)) return SV_ERR_ALIGN;
  Params p{};
  Geometry g;
  if (!fill_geometry(p, V, dtype, &g)) return SV_ERR_SHAPE;
  p.rows0 = logits;
  p.temp = temperature;
  p.topk = top_k;
  p.topp = top_p;
  p.seed = philox_seed;
  p.offset = philox_offset;
  p.B = B;
  p.K = K;
  p.nunits = B * K;
  p.bulk_ok = ((V * es) % 16 == 0) && aligned(logits, 16);
  p.out_tokens = out_tokens;
  return do_launch(MODE_SAMPLE, dtype, p, g, static_cast<cudaStream_t>(stream));
}

sv_status spec_philox_uniforms(uint64_t philox_seed, uint64_t philox_offset, int B, int K1,
                               uint32_t* out, void* stream) {
  if (B < 1 || K1 < 1 || (long long)B * K1 > (1ll << 26)) return SV_ERR_SHAPE;
  if (!out) return SV_ERR_NULL;
  if (!aligned(out, 4)) return SV_ERR_ALIGN;
  const int n = B * K1;
  philox_kernel<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      philox_seed, philox_offset, B, K1, out);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

const char* sv_status_string(sv_status status) {
  switch (status) {
    case SV_OK: return "ok";
    case SV_ERR_NULL: return "a required pointer is NULL";
    case SV_ERR_SHAPE: return "B, K, R or V outside the supported limits";
    case SV_ERR_DTYPE: return "unknown logit dtype";
    case SV_ERR_WORKSPACE: return "workspace too small or not 16-byte aligned";
    case SV_ERR_CUDA: return "CUDA launch or attribute call failed";
    case SV_ERR_ALIGN: return "pointer not aligned to its element size";
    case SV_ERR_SCRATCH: return "batch needs more workspace than spec_verify_noalloc's fixed scratch";
  }
  return "unknown status";
}

int sv_version(void) { return 200; }

#ifdef SV_TRACE
int sv_trace_copy(unsigned long long* host, size_t n) {
  return (int)cudaMemcpyFromSymbol(host, sv::g_trace, n * sizeof(unsigned long long));
}
#endif

}  // extern "C"
