// spec_verify.cu -- verify-and-sample kernels for GB300 (sm_103a) and the C ABI.
//
// Work decomposition. A "unit" is one (sequence b, position i) pair, i in
// [0, K]: for i < K it owns target row i and draft row i, for i == K the
// target row K (bonus position). One thread-block cluster of C CTAs serves one
// unit; CTA c holds the vocabulary slice [c*slice, (c+1)*slice) of the unit's
// rows in shared memory, loaded once from HBM by bulk copies. Every later pass
// (row maximum, truncation threshold search, probabilities of the draft token,
// inverse-CDF scan) reads shared memory only; CTAs combine partial results
// through distributed shared memory.
//
// Method (see the pages cited in include/spec_verify.h): temperature scaling,
// matched top-k / top-p truncation of target and draft, acceptance with
// min(1, p/q) in order, replacement from (p - q)+ or the bonus token from p_K,
// greedy argmax-prefix matching at temperature 0.
//
// Truncation: the kept set is a prefix of the order (logit desc, id asc). Its
// last key is found by radix selection over order-preserving 32-bit keys, 8
// bits per level (two levels for bf16 logits, four for fp32), counting tokens
// for top-k and fixed-point mass for top-p. Only tokens that provably can be in
// the kept set take part: for top-k, tokens at or above the largest per-CTA
// k-th largest per-thread maximum (each CTA alone holds k tokens at least that
// large); for top-p alone, tokens within ln(V / (1 - top_p)) of the maximum in
// temperature-scaled units (all other tokens together weigh less than
// (1 - top_p) times the maximum's weight). Ties at the cut are split by token
// id with an id-ordered count across the cluster.
//
// Sums: weights e = exp((z - max)/T) in fp32 are converted to fixed point
// floor(e * 2^S) with S = 63 - ceil(log2 V); all sums are exact 64-bit integer
// sums, so the kernels are deterministic and order-independent, and the
// inverse-CDF decision C_j * 2^24 > k_v * S_total is taken exactly on those
// integers. Residual weights (p - q)+ are fp32 and enter the scan as
// floor(r * 2^62).

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
  int nlev;                 // radix levels: 2 (bf16) or 4 (fp32)
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

// One row's values shared by every CTA of the cluster after the exchanges.
struct RowInfo {
  float m, zmin;
  int argmax;
  int bad;
  uint32_t tau;             // eligibility key threshold for the selection
  uint32_t thr;             // kept: key > thr, or key == thr and id <= tie
  int tie;
  int pad;
  unsigned long long ZL;    // kept mass (fixed point)
  unsigned long long zfar;  // fixed-point mass of non-eligible tokens (top-p only rows)
};

struct XSlot {               // per-row payload of one cluster exchange
  float best;
  int best_id;
  float zmin;
  int bad;
  uint32_t kth;
  uint32_t pad;
  unsigned long long a, b;
};

struct Work {
  unsigned long long mbar;
  unsigned long long pad0;
  XSlot xch[2][2];                          // [buffer][row]
  unsigned long long hmass[2][2][256];      // [buffer][row][digit]
  unsigned int hcnt[2][2][256];
  unsigned long long gmass[2][256];         // cluster-wide histogram of the current level
  unsigned int gcnt[2][256];
  unsigned long long scan64[NWARP];
  unsigned int scan32[NWARP];
  unsigned int kthh[2][256];                // per-CTA pool selection histogram
  RowInfo row[2];
  int bcast_i[8];
  unsigned long long bcast_u[4];
  double bcast_d[4];
};

// Order key restricted to the bits a logit of this dtype can set. For bf16 the
// low 16 bits of okey() are all zeros (positive) or all ones (negative), so
// they are dropped; the radix levels then build exactly these masked keys.
__device__ __forceinline__ uint32_t mkey(float z, uint32_t mask) { return okey(z) & mask; }
// Float value of a masked key (inverse of mkey on values of the dtype).
__device__ __forceinline__ float mkey_to_float(uint32_t k, uint32_t mask) {
  return key_to_float((k & 0x80000000u) ? k : (k | ~mask));
}

template <typename DT>
__device__ __forceinline__ float ld_elem(const DT* d, int j) {
  return to_f32<DT>(d[j]);
}
template <typename DT>
__device__ __forceinline__ float ld_peer_elem(const DT* d, int j, uint32_t rank);
template <>
__device__ __forceinline__ float ld_peer_elem<float>(const float* d, int j, uint32_t rank) {
  return ld_peer_f32(d + j, rank);
}
template <>
__device__ __forceinline__ float ld_peer_elem<__nv_bfloat16>(const __nv_bfloat16* d, int j,
                                                             uint32_t rank) {
  const uint16_t h = ld_peer_u16(d + j, rank);
  return __uint_as_float(((uint32_t)h) << 16);
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
    // warp 0 scans digits from 255 down
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
        if (l == 0) scratch[0] = 0xffffffffu;  // not enough valid keys
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
// Cluster-wide digit histogram -> digit where the cumulative (from the top)
// count or mass first reaches the target. Runs on warp `r` for row r.
struct DigitPick {
  int digit;
  unsigned int cnt_above;           // count of tokens in larger digits
  unsigned long long mass_above;    // mass of tokens in larger digits
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
  int nacc = P.K, bad = 0, last = -1;
  const volatile unsigned long long* u = P.ws_units + (size_t)b * (P.K + 1);
  for (int q = 0; q <= P.K; ++q) {
    const unsigned long long rec = u[q];
    bad |= (int)((rec >> 33) & 1ull);
    if (q < P.K && nacc == P.K && !((rec >> 32) & 1ull)) nacc = q;
  }
  last = (int)(uint32_t)u[nacc];
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
template <typename DT, int MODE>
__global__ void __launch_bounds__(NT, 1) sv_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t C = cluster_size();
  const uint32_t rank = cluster_rank();
  const int unit = blockIdx.x / C;
  const int tid = threadIdx.x;
  const int V = P.V;
  const int es = (int)sizeof(DT);
  const size_t row_bytes = ((size_t)P.slice * es + 15) & ~(size_t)15;
  DT* data[2] = {reinterpret_cast<DT*>(smem), reinterpret_cast<DT*>(smem + row_bytes)};
  Work& W = *reinterpret_cast<Work*>(smem + 2 * row_bytes);

  // ---------------------------------------------------------------- unit
  int b, i, nrows, seq;
  const DT* gro[2] = {nullptr, nullptr};
  if (MODE == MODE_VERIFY) {
    b = unit / (P.K + 1);
    i = unit % (P.K + 1);
    seq = b;
    gro[0] = reinterpret_cast<const DT*>(P.rows0) + ((size_t)b * (P.K + 1) + i) * V;
  } else if (MODE == MODE_SAMPLE) {
    b = unit / P.K;
    i = unit % P.K;
    seq = b;
    gro[0] = reinterpret_cast<const DT*>(P.rows0) + (size_t)unit * V;
  } else {
    b = unit;
    i = 0;
    seq = unit;
    gro[0] = reinterpret_cast<const DT*>(P.rows0) + (size_t)unit * V;
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
  nrows = 1;
  if (MODE == MODE_VERIFY && i < P.K && !greedy && !param_bad) {
    if (P.rows1 == nullptr) {
      param_bad = true;
    } else {
      nrows = 2;
      gro[1] = reinterpret_cast<const DT*>(P.rows1) + ((size_t)b * P.K + i) * V;
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
        const char* src = reinterpret_cast<const char*>(gro[r] + v0);
        char* dst = reinterpret_cast<char*>(data[r]);
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
    for (int r = 0; r < nrows; ++r)
      for (int j = tid; j < n; j += NT) data[r][j] = gro[r][v0 + j];
    __syncthreads();
  }

  SV_MARK(1);
  const int j0 = tid * P.ept;
  const int j1 = min(n, j0 + P.ept);

  // ------------------------------------------- pass A: max, argmax, min, NaN
  float best[2], zmn[2];
  int bidx[2], bad[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    best[r] = -INFINITY;
    zmn[r] = INFINITY;
    bidx[r] = 0x7fffffff;
    bad[r] = 0;
    if (r < nrows) {
      for (int j = j0; j < j1; ++j) {
        const float z = ld_elem<DT>(data[r], j);
        if (!(z <= 3.402823466e38f)) bad[r] = 1;      // NaN or +inf
        if (z > best[r]) {
          best[r] = z;
          bidx[r] = j;
        }
        zmn[r] = fminf(zmn[r], z);
      }
    }
  }
  const bool topk_on = topk > 0 && topk < V;
  const int kk = topk_on ? topk : V;
  // per-CTA k-th largest per-thread maximum (top-k eligibility bound)
  uint32_t kth[2] = {KEY_ALL, KEY_ALL};
  if (!greedy && topk_on && kk <= NT) {
    for (int r = 0; r < nrows; ++r)
      kth[r] = block_kth_largest(mkey(best[r], P.keymask), j1 > j0, kk, W.kthh[r], W.scan32, P.nlev);
  }
  // block reductions (deterministic butterflies)
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    for (int o = 16; o; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best[r], o);
      const int oi = __shfl_xor_sync(0xffffffffu, bidx[r], o);
      if (ob > best[r] || (ob == best[r] && oi < bidx[r])) {
        best[r] = ob;
        bidx[r] = oi;
      }
      zmn[r] = fminf(zmn[r], __shfl_xor_sync(0xffffffffu, zmn[r], o));
      bad[r] |= __shfl_xor_sync(0xffffffffu, bad[r], o);
    }
  }
  {
    __shared__ float sb[2][NWARP], sz[2][NWARP];
    __shared__ int si[2][NWARP], sbad[2][NWARP];
    if (lane_id() == 0)
      for (int r = 0; r < 2; ++r) {
        sb[r][warp_id()] = best[r];
        si[r][warp_id()] = bidx[r];
        sz[r][warp_id()] = zmn[r];
        sbad[r][warp_id()] = bad[r];
      }
    __syncthreads();
    if (tid < 2) {
      const int r = tid;
      float bb = -INFINITY, zz = INFINITY;
      int ii = 0x7fffffff, bd = load_bad;
      for (int w = 0; w < NWARP; ++w) {
        if (sb[r][w] > bb || (sb[r][w] == bb && si[r][w] < ii)) {
          bb = sb[r][w];
          ii = si[r][w];
        }
        zz = fminf(zz, sz[r][w]);
        bd |= sbad[r][w];
      }
      XSlot& x = W.xch[0][r];
      x.best = bb;
      x.best_id = (ii == 0x7fffffff) ? 0x7fffffff : v0 + ii;
      x.zmin = zz;
      x.bad = bd;
      x.kth = kth[r];
    }
  }
  __syncthreads();
  SV_MARK(2);
  cluster_sync();  // X1
  SV_MARK(3);
  if (tid < 2) {
    const int r = tid;
    float bb = -INFINITY, zz = INFINITY;
    int ii = 0x7fffffff, bd = 0;
    uint32_t kt = KEY_ALL;
    for (uint32_t c = 0; c < C; ++c) {
      const float pb = ld_peer_f32(&W.xch[0][r].best, c);
      const int pi = (int)ld_peer_u32(&W.xch[0][r].best_id, c);
      if (pb > bb || (pb == bb && pi < ii)) {
        bb = pb;
        ii = pi;
      }
      zz = fminf(zz, ld_peer_f32(&W.xch[0][r].zmin, c));
      bd |= (int)ld_peer_u32(&W.xch[0][r].bad, c);
      kt = max(kt, ld_peer_u32(&W.xch[0][r].kth, c));
    }
    RowInfo& ri = W.row[r];
    ri.m = bb;
    ri.zmin = zz;
    ri.argmax = ii;
    ri.bad = bd | (bb == -INFINITY ? 1 : 0);
    ri.tau = kt;
    ri.thr = KEY_ALL;
    ri.tie = NO_TIE;
    ri.ZL = 0;
    ri.zfar = 0;
  }
  __syncthreads();

  bool unit_err = param_bad || W.row[0].bad || (nrows == 2 && W.row[1].bad);
  int xbuf = 1;  // next exchange buffer

  // --------------------------------------------------------- greedy / error
  if (greedy || unit_err) {
    if (rank == 0 && tid == 0) {
      const int am = W.row[0].argmax;
      if (MODE == MODE_VERIFY) {
        // published after the cluster barrier below
      } else if (MODE == MODE_SAMPLE) {
        P.out_tokens[unit] = unit_err ? -1 : am;
      }
    }
    if (MODE == MODE_PROBS) {
      float* out = P.out_probs + (size_t)unit * V + v0;
      const int am = W.row[0].argmax;
      for (int j = tid; j < n; j += NT)
        out[j] = unit_err ? __int_as_float(0x7fc00000) : ((v0 + j == am) ? 1.0f : 0.0f);
    }
    cluster_sync();  // peers may still read this CTA's exchange slots
    if (MODE == MODE_VERIFY && rank == 0 && tid == 0) {
      const int am = W.row[0].argmax;
      publish_unit(P, unit, b, unit_err ? -1 : am, !unit_err && i < P.K && dtok == am, unit_err);
    }
    if (load_bad) mbar_wait_bounded(&W.mbar, 0, WAIT_LIMIT_NS);
    return;
  }

  // ------------------------------------------------------------ sampling
  RowScale sc[2];
  for (int r = 0; r < 2; ++r) sc[r] = make_scale(W.row[r].m, T);
  const bool topp_on = topp < 1.0f;
  const float fscale = P.fix_scale;

  // eligibility for top-p alone: z >= m - (ln(V/(1-P)) + margin) * T
  if (!topk_on && topp_on && tid < 2) {
    const int r = tid;
    const double tau_d = log((double)V / (1.0 - (double)topp)) + 0.05;
    const float zt = (float)((double)W.row[r].m - tau_d * (double)T);
    W.row[r].tau = (zt > W.row[r].zmin && isfinite(zt)) ? mkey(zt, P.keymask) : KEY_ALL;
  }
  if (!topk_on && !topp_on && tid < 2) W.row[tid].tau = KEY_ALL;
  __syncthreads();

  // ----------------------------------------------- radix selection stages
  // Stage 0: top-k (count); stage 1: top-p (mass). Both rows in lockstep.
  uint32_t tk[2] = {0, 0};
  unsigned int jk[2] = {0, 0};
  unsigned long long Etk[2] = {0, 0};
  double Z1[2] = {0, 0};
  uint32_t thr[2] = {KEY_ALL, KEY_ALL};
  unsigned int jt[2] = {0, 0}, neq_all[2] = {0, 0};
  unsigned long long ZL[2] = {0, 0};
  bool need_tie[2] = {false, false};
  const bool any_sel = topk_on || topp_on;

  for (int stage = 0; stage < 2 && any_sel; ++stage) {
    const bool by_mass = (stage == 1);
    if (stage == 0 && !topk_on) continue;
    if (stage == 1 && !topp_on) continue;
    uint32_t prefix[2] = {0, 0}, pmask = 0;
    unsigned int cabove[2] = {0, 0};
    unsigned long long mabove[2] = {0, 0};
    double need_m[2] = {0, 0};
    unsigned int lastcnt[2] = {0, 0};
    // Top-p over the whole row: a first level of 256 linear bins in
    // temperature-scaled distance from the maximum, d = (m - z)/T in
    // [0, ln(V/(1-top_p))], spreads flat rows over many bins (key bytes would
    // put them in a handful). Later levels refine exact keys inside the bin.
    const bool use_dbin = (stage == 1 && !topk_on);
    const float dscale =
        use_dbin ? (float)(256.0 / (log((double)V / (1.0 - (double)topp)) + 0.05)) : 0.f;
    int dsel[2] = {-1, -1};
    auto dbin = [&](float z, int r) -> int {
      const float d = (sc[r].m - z) * sc[r].inv_hi;
      return min(255, (int)(d * dscale));
    };
    const int nl = P.nlev + (use_dbin ? 1 : 0);
    for (int lev = 0; lev < nl; ++lev) {
      const bool dlev = use_dbin && lev == 0;
      const int shift = 24 - 8 * (lev - (use_dbin ? 1 : 0));
      const int buf = xbuf;
      xbuf ^= 1;
      for (int t = tid; t < 2 * 256; t += NT) {
        W.hcnt[buf][t >> 8][t & 255] = 0;
        W.hmass[buf][t >> 8][t & 255] = 0;
      }
      __syncthreads();
      float zfar_t[2] = {0.f, 0.f};
      for (int r = 0; r < nrows; ++r) {
        const uint32_t tau = W.row[r].tau;
        for (int j = j0; j < j1; ++j) {
          const float z = ld_elem<DT>(data[r], j);
          const uint32_t key = mkey(z, P.keymask);
          bool in;
          if (stage == 0) {
            in = key >= tau;
          } else if (topk_on) {
            in = key > tk[r];                     // the tie group at tk enters as one pseudo token
          } else {
            in = key >= tau;
            if (!in && lev == 0) zfar_t[r] += weight_fast(z, sc[r]);
          }
          if (in && use_dbin && !dlev) in = dbin(z, r) == dsel[r];
          if (in && (key & pmask) == prefix[r]) {
            const unsigned int dg = dlev ? 255u - (unsigned int)dbin(z, r) : (key >> shift) & 255u;
            atomicAdd(&W.hcnt[buf][r][dg], 1u);
            const unsigned long long E = to_fixed(weight(z, sc[r]), fscale);
            if (E) atomicAdd(&W.hmass[buf][r][dg], E);
          }
        }
      }
      if (stage == 1 && topk_on && rank == 0 && tid < nrows) {
        const int r = tid;                          // pseudo token: the j_k kept members of tie group tk
        if ((tk[r] & pmask) == prefix[r]) {
          const unsigned int dg = (tk[r] >> shift) & 255u;
          atomicAdd(&W.hcnt[buf][r][dg], jk[r]);
          atomicAdd(&W.hmass[buf][r][dg], (unsigned long long)jk[r] * Etk[r]);
        }
      }
      if (stage == 1 && !topk_on && lev == 0) {
        for (int r = 0; r < nrows; ++r) {
          const unsigned long long zf = block_sum<unsigned long long>(
              (unsigned long long)to_fixed(zfar_t[r], fscale), W.scan64);
          if (tid == 0) W.xch[buf][r].a = zf;
        }
      }
      __syncthreads();
      SV_MARK(10 + 2 * stage);
      cluster_sync();
      SV_MARK(11 + 2 * stage);
      // cluster-wide histogram: thread t -> row t>>8, digit t&255
      {
        const int r = tid >> 8, dg = tid & 255;
        if (r < nrows) {
          unsigned int c = 0;
          unsigned long long w = 0;
          for (uint32_t q = 0; q < C; ++q) {
            c += ld_peer_u32(&W.hcnt[buf][r][dg], q);
            w += ld_peer_u64(&W.hmass[buf][r][dg], q);
          }
          W.gcnt[r][dg] = c;
          W.gmass[r][dg] = w;
        }
        if (stage == 1 && !topk_on && lev == 0 && tid < nrows) {
          unsigned long long zf = 0;
          for (uint32_t q = 0; q < C; ++q) zf += ld_peer_u64(&W.xch[buf][tid].a, q);
          W.row[tid].zfar = zf;
        }
      }
      __syncthreads();
      if (stage == 1 && lev == 0) {
        for (int r = 0; r < nrows; ++r) {
          if (!topk_on) {
            // Z1 = every eligible token's mass + the far tail
            unsigned long long s = 0;
            for (int dg = 0; dg < 256; ++dg) s += W.gmass[r][dg];
            Z1[r] = (double)(s + W.row[r].zfar);
          }
          need_m[r] = (double)topp * Z1[r];
        }
      }
      if (warp_id() < nrows) {
        const int r = warp_id();
        const unsigned int need_c = stage == 0 ? (unsigned int)kk - cabove[r] : 0u;
        const DigitPick pk = pick_digit(W.gcnt[r], W.gmass[r], by_mass, need_c,
                                        need_m[r] - (double)mabove[r]);
        if (lane_id() == 0) {
          W.bcast_i[r] = pk.digit;
          W.bcast_i[2 + r] = (int)pk.cnt_above;
          W.bcast_u[r] = pk.mass_above;
          W.bcast_i[4 + r] = (int)W.gcnt[r][pk.digit];
        }
      }
      __syncthreads();
      for (int r = 0; r < nrows; ++r) {
        if (dlev)
          dsel[r] = 255 - W.bcast_i[r];
        else
          prefix[r] |= (uint32_t)W.bcast_i[r] << shift;
        cabove[r] += (unsigned int)W.bcast_i[2 + r];
        mabove[r] += W.bcast_u[r];
        lastcnt[r] = (unsigned int)W.bcast_i[4 + r];
      }
      if (!dlev) pmask |= 255u << shift;
      __syncthreads();
    }
    // stage result
    for (int r = 0; r < nrows; ++r) {
      const unsigned long long Et = to_fixed(weight(mkey_to_float(prefix[r], P.keymask), sc[r]), fscale);
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
        double jf = Et > 0 ? ceil(gap / (double)Et) : 1.0;
        unsigned int j = (unsigned int)fmax(1.0, fmin(jf, (double)lastcnt[r]));
        thr[r] = prefix[r];
        jt[r] = j;
        neq_all[r] = (topk_on && prefix[r] == tk[r]) ? neq_all[r] : lastcnt[r];
        ZL[r] = mabove[r] + (unsigned long long)j * Et;
      }
    }
  }

  SV_MARK(4);
  // ---------------------------------------------------- tie split by token id
  for (int r = 0; r < nrows; ++r) need_tie[r] = any_sel && jt[r] < neq_all[r];
  if (need_tie[0] || need_tie[1]) {
    unsigned int cnt[2] = {0, 0};
    for (int r = 0; r < nrows; ++r)
      if (need_tie[r])
        for (int j = j0; j < j1; ++j) cnt[r] += (mkey(ld_elem<DT>(data[r], j), P.keymask) == thr[r]);
    unsigned int excl[2], tot[2];
    for (int r = 0; r < 2; ++r) excl[r] = block_excl_scan<unsigned int>(cnt[r], W.scan32, &tot[r]);
    const int buf = xbuf;
    xbuf ^= 1;
    if (tid == 0) {
      W.xch[buf][0].kth = tot[0];
      W.xch[buf][1].kth = tot[1];
    }
    __syncthreads();
    cluster_sync();
    int found[2] = {NO_TIE, NO_TIE};
    for (int r = 0; r < nrows; ++r) {
      if (!need_tie[r]) continue;
      unsigned int off = 0;
      for (uint32_t q = 0; q < rank; ++q) off += ld_peer_u32(&W.xch[buf][r].kth, q);
      const unsigned int target = jt[r] - 1;      // 0-indexed position in the tie group
      const unsigned int lo = off + excl[r];
      if (cnt[r] > 0 && target >= lo && target < lo + cnt[r]) {
        unsigned int seen = lo;
        for (int j = j0; j < j1; ++j)
          if (mkey(ld_elem<DT>(data[r], j), P.keymask) == thr[r]) {
            if (seen == target) {
              found[r] = v0 + j;
              break;
            }
            ++seen;
          }
      }
    }
    const int buf2 = xbuf;
    xbuf ^= 1;
    if (tid < 2) W.xch[buf2][tid].best_id = NO_TIE;
    __syncthreads();
    for (int r = 0; r < nrows; ++r)
      if (found[r] != NO_TIE) W.xch[buf2][r].best_id = found[r];
    __syncthreads();
    cluster_sync();
    if (tid < nrows) {
      int f = NO_TIE;
      for (uint32_t q = 0; q < C; ++q) f = min(f, (int)ld_peer_u32(&W.xch[buf2][tid].best_id, q));
      W.bcast_i[6 + tid] = f;
    }
    __syncthreads();
  }
  if (tid < nrows) {
    W.row[tid].thr = thr[tid];
    W.row[tid].tie = need_tie[tid] ? W.bcast_i[6 + tid] : NO_TIE;
  }
  __syncthreads();
  int tie[2] = {W.row[0].tie, W.row[1].tie};
  for (int r = 0; r < 2; ++r) thr[r] = W.row[r].thr;

  SV_MARK(5);
  // -------------------------------------- full support: exact normaliser
  const bool need_norm = !any_sel && (MODE == MODE_PROBS || (MODE == MODE_VERIFY && i < P.K));
  if (need_norm) {
    unsigned long long s[2] = {0, 0};
    for (int r = 0; r < nrows; ++r)
      for (int j = j0; j < j1; ++j) s[r] += to_fixed(weight(ld_elem<DT>(data[r], j), sc[r]), fscale);
    unsigned long long tot[2];
    for (int r = 0; r < 2; ++r) tot[r] = block_sum<unsigned long long>(s[r], W.scan64);
    const int buf = xbuf;
    xbuf ^= 1;
    if (tid == 0) {
      W.xch[buf][0].a = tot[0];
      W.xch[buf][1].a = tot[1];
    }
    __syncthreads();
    cluster_sync();
    for (int r = 0; r < nrows; ++r) {
      unsigned long long z = 0;
      for (uint32_t q = 0; q < C; ++q) z += ld_peer_u64(&W.xch[buf][r].a, q);
      ZL[r] = z;
    }
  }

  const uint32_t kmask = P.keymask;
  auto kept = [&](int r, float z, int id) -> bool {
    const uint32_t key = mkey(z, kmask);
    return key > thr[r] || (key == thr[r] && id <= tie[r]);
  };

  // --------------------------------------------------- probabilities hook
  if (MODE == MODE_PROBS) {
    float* out = P.out_probs + (size_t)unit * V + v0;
    const double inv = 1.0 / (double)ZL[0];
    for (int j = tid; j < n; j += NT) {
      const float z = ld_elem<DT>(data[0], j);
      float pr = 0.0f;
      if (kept(0, z, v0 + j)) pr = (float)((double)to_fixed(weight(z, sc[0]), fscale) * inv);
      out[j] = pr;
    }
    cluster_sync();
    return;
  }

  SV_MARK(6);
  // ------------------------------------------------------------ acceptance
  bool flag = false;
  if (MODE == MODE_VERIFY && i < P.K) {
    const uint32_t owner = (uint32_t)(dtok / P.slice);
    const int jj = dtok - (int)owner * P.slice;
    double pq[2];
    for (int r = 0; r < 2; ++r) {
      const float z = ld_peer_elem<DT>(data[r], jj, owner);
      pq[r] = kept(r, z, dtok)
                  ? (double)to_fixed(weight(z, sc[r]), fscale) / (double)ZL[r]
                  : 0.0;
    }
    uint32_t ku, kv;
    philox_uniform_bits(P.seed, P.offset, (uint32_t)b, (uint32_t)i, &ku, &kv);
    flag = (double)ku * 5.9604644775390625e-08 * pq[1] < pq[0];
  }

  SV_MARK(7);
  // ------------------------------------------- inverse-CDF in token-id order
  uint32_t ku, kv;
  philox_uniform_bits(P.seed, P.offset, (uint32_t)b, (uint32_t)i, &ku, &kv);
  const bool residual = (MODE == MODE_VERIFY && i < P.K);
  const float sp = residual ? (float)((double)fscale / (double)ZL[0]) : 0.f;
  const float sq = residual ? (float)((double)fscale / (double)ZL[1]) : 0.f;
  auto wgt = [&](int j, bool res) -> unsigned long long {
    const float z = ld_elem<DT>(data[0], j);
    if (!kept(0, z, v0 + j)) return 0ull;
    const float ep = weight(z, sc[0]);
    if (!res) return to_fixed(ep, fscale);
    const float zq = ld_elem<DT>(data[1], j);
    // rounded products and difference (no FMA contraction): identical rows give d == 0
    const float q = kept(1, zq, v0 + j) ? __fmul_rn(weight(zq, sc[1]), sq) : 0.0f;
    const float d = __fsub_rn(__fmul_rn(ep, sp), q);
    return d > 0.0f ? __float2ull_rz(d * 4611686018427387904.0f) : 0ull;
  };
  bool use_res = residual;
  for (int attempt = 0; attempt < 2; ++attempt) {
    unsigned long long s = 0;
    for (int j = j0; j < j1; ++j) s += wgt(j, use_res);
    unsigned long long ctot;
    const unsigned long long texcl = block_excl_scan<unsigned long long>(s, W.scan64, &ctot);
    const int buf = xbuf;
    xbuf ^= 1;
    if (tid == 0) W.xch[buf][0].a = ctot;
    __syncthreads();
    cluster_sync();
    unsigned long long off = 0, S = 0;
    for (uint32_t q = 0; q < C; ++q) {
      const unsigned long long t = ld_peer_u64(&W.xch[buf][0].a, q);
      if (q < rank) off += t;
      S += t;
    }
    if (S == 0 && use_res) {       // (p - q)+ has no mass: sample from p
      use_res = false;
      continue;
    }
    const unsigned long long lo = off + texcl, hi = lo + s;
    const unsigned long long kvs = (unsigned long long)kv;
    // this thread holds the first token whose inclusive CDF exceeds v * S
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
      if (MODE == MODE_SAMPLE) {
        P.out_tokens[unit] = tok;
      } else {
        publish_unit(P, unit, b, tok, flag, false);
      }
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
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
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

static Geometry geometry(int V, int es) {
  Geometry g{};
  const size_t budget = 110 * 1024;     // two CTAs per SM when it fits
  const size_t hard = 227 * 1024;
  for (int C = 1; C <= 16; C *= 2) {
    int slice = (V + C - 1) / C;
    slice = (slice + 15) & ~15;
    const size_t rb = ((size_t)slice * es + 15) & ~(size_t)15;
    const size_t smem = 2 * rb + sizeof(Work);
    g.C = C;
    g.slice = slice;
    g.smem = smem;
    if (smem <= budget || (C == 8 && smem <= hard) || C == 16) break;
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

static void fill_geometry(Params& p, int V, sv_dtype dt, Geometry* g) {
  const int es = dt == SV_BF16 ? 2 : 4;
  *g = geometry(V, es);
  p.V = V;
  p.slice = g->slice;
  p.ept = g->ept;
  p.nlev = dt == SV_BF16 ? 2 : 4;
  p.keymask = dt == SV_BF16 ? 0xFFFF0000u : 0xFFFFFFFFu;
  p.fix_scale = ldexpf(1.0f, fix_scale_shift(V));
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
  fill_geometry(p, V, dtype, &g);
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
  fill_geometry(p, V, dtype, &g);
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
  fill_geometry(p, V, dtype, &g);
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
  }
  return "unknown status";
}

int sv_version(void) { return 100; }

#ifdef SV_TRACE
int sv_trace_copy(unsigned long long* host, size_t n) {
  return (int)cudaMemcpyFromSymbol(host, sv::g_trace, n * sizeof(unsigned long long));
}
#endif

}  // extern "C"
