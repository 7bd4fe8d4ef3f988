// spec_verify.cu -- verify-and-sample kernels for GB300 (sm_103a) and the C ABI.
//
// Method (pages cited in include/spec_verify.h): temperature scaling, matched
// top-k / top-p truncation of target and draft rows, acceptance with min(1, p/q)
// in order, replacement from (p - q)+ or the bonus token from p_K, and greedy
// argmax-prefix matching at temperature 0.
//
// Work decomposition. A "unit" is one (sequence b, position i): for i < K the
// target row i and the draft row i (one row at temperature 0), for i == K the
// target row K. A persistent thread-block cluster of C CTAs walks a strided
// share of the units; CTA r holds the vocabulary slice [r*slice, (r+1)*slice)
// of a unit's rows in shared memory. Row slices arrive by bulk copies (the TMA
// engine) into a ring of slots that is filled one or more units ahead, so the
// next unit's rows stream in while the current one is computed. Every logit
// leaves HBM once; CTAs combine partial results through distributed shared
// memory (DSMEM) at a few cluster barriers per unit.
//
// Per sampling row:
//   A  the slice maximum (packed bf16x2 max; NaN/+inf detection).
//   B  weights e = 2^(z*c - R), c = log2(e)/T, in a CTA-local frame R (an even
//      integer >= the slice maximum * c), summed per thread into 16 bins of two
//      binades of e each (bin = the exponent of e, no atomics), then reduced to
//      exact 64-bit fixed-point bin masses. Frames differ between CTAs by a
//      whole number of bins, so the cluster merges bins by shifting.
//      Top-k rows (k <= 256) instead list the tokens at or above the CTA's
//      k-th largest per-thread maximum (each CTA alone holds k tokens that
//      large, so the listed tokens contain the top k).
//   S1 cluster exchange: maxima, frames, bins or list sizes.
//   the bin holding the top-p cut is refined over logit keys (256 sub-bins per
//      level, one level for bf16 in practice) until one logit value remains;
//      its run of equal logits is split by token id.                    [S2..]
//   D  acceptance in the CTA that owns the drafted token; the residual
//      (p - q)+ or bonus p summed in token-id order per thread.          [S3]
//      The CTA holding the crossing of v * total finds the token.
//
// Sums that decide a token (normaliser, cut, inverse CDF) are exact integer
// sums of fixed-point weights, independent of summation order; identical target
// and draft rows give identical p and q.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include <thread>

#include "../../include/spec_verify.h"
#include "launch_cache.h"
#include "sv_device.cuh"

namespace sv {

enum { MODE_VERIFY = 0, MODE_PROBS = 1, MODE_SAMPLE = 2 };

constexpr int NB = 16;          // mass bins (two binades of the weight each)
constexpr int NSUB = 256;       // sub-bins of one refinement level
constexpr int LC = 512;         // listed top-k candidates per CTA and row
constexpr int GCAP = 1024;      // gathered top-k candidates per row
constexpr int KFAST = 256;      // largest top_k served by the candidate lists
constexpr int MAXLEV = 8;       // refinement levels before giving up (error)
constexpr int MR = 32;          // unit metadata ring
constexpr int NSMAX = 4;        // row slots
constexpr int FIX = 44;         // fixed-point weights: floor(e * 2^44)

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

// X1 row flags
constexpr uint32_t F_NAN = 1u, F_PINF = 2u, F_EXTREME = 4u, F_OVER = 8u;

struct KhRow;

struct Params {
  const void* rows0;            // target [B][K+1][V] | probs rows [R][V] | draft [B][K][V]
  const void* rows1;            // draft [B][K][V] (verify)
  const int32_t* dtok;          // [B][K]
  const float* temp;
  const int32_t* topk;
  const float* topp;
  uint64_t seed, offset;
  int B, K, V, nunits;
  int C, slice, ept, slot_elems, NS;
  int bulk_ok;
  int32_t* out_tokens;          // verify [B][K+1]; sample [B][K]
  int32_t* out_n;
  float* out_probs;
  unsigned long long* ws_units; // per unit: bits 0..31 token, bit 32 flag, bit 33 error
  unsigned int* ws_tickets;     // per sequence
  unsigned int* ws_error;       // bit 0 = a bulk copy did not complete in time (cleared at the call's end)
  unsigned long long* ws_best;  // greedy rows: (okey(max) << 32) | ~argmax
  unsigned int* ws_rcnt;        // [0]: greedy_kernel CTAs finished
  unsigned int* ws_rflag;       // greedy rows: NaN / +inf seen
  unsigned int* ws_work;        // set by greedy_kernel when other units exist
  unsigned int* ws_done;        // cluster-kernel CTAs finished (resets ws_work)
  int greedy_split;             // temperature-0 verify units go to greedy_kernel
  int greedy_only;              // no draft logits: greedy_kernel serves the whole batch
  int fast_split;               // sampled sequences go to keyhist_kernel (bf16) or fstream_kernel (fp32)
  KhRow* ws_rowres;             // keyhist_kernel: per-row results [B][2K+1]
  unsigned int* ws_fb;          // keyhist_kernel: 1 = sequence handed to the cluster kernel
  unsigned int* ws_fnext;       // keyhist_kernel: work counter
  unsigned int* ws_fdone;       // keyhist_kernel: CTAs finished
  uint32_t* ws_lists;           // keyhist_kernel: kept-token ids of target rows [B][K+1][256]
  int* ws_perm;                 // fstream_kernel: sequences in processing order [B]
  const uint64_t* offset_ptr;   // Philox offset in device memory (spec_verify_step), else NULL
};

// The Philox offset of this call: from device memory when the step keeps it there.
__device__ __forceinline__ uint64_t philox_offset_of(const Params& P) {
  return P.offset_ptr ? __ldcg(reinterpret_cast<const unsigned long long*>(P.offset_ptr)) : P.offset;
}

struct Meta {
  float T, P;
  int k, d;
  int g;                        // the unit's sequence is on the greedy path
  int pad[3];
};

// Exchanged through DSMEM after the first cluster barrier of a unit.
struct X1Row {
  float m;                // CTA maximum (raw logit), -inf when none is finite
  uint32_t flags;         // F_*
  float R;                // CTA frame
  uint32_t ncand;         // listed top-k candidates
  unsigned long long best;  // (okey(max) << 32) | ~argmax  (greedy)
  unsigned long long bins[NB];
  uint32_t cnts[NB];
};
struct X3 {
  unsigned long long R, P;  // residual and target mass of this CTA (fixed 2^-40)
  uint32_t flag;            // acceptance flag (owner CTA of the drafted token)
  uint32_t pad;
};
// One refinement level of one row: counts and masses per sub-bin.
struct X2Row {
  uint32_t cnt[NSUB];
  unsigned long long mass[NSUB];
};

enum { ST_DONE = 0, ST_KEYS = 1 };
enum { T_MASS = 0, T_COUNT = 1 };
enum { RM_ALL = 0, RM_TOPP = 1, RM_LIST = 2, RM_GENERAL = 3 };

// Cluster-wide state of one row of the current unit (identical in every CTA
// except the fields marked local).
struct RowG {
  float c;                // log2(e)/T (rounded)
  float Rg;               // cluster frame
  float mg;               // cluster maximum
  float Rl;               // local: this CTA's frame
  int sh;                 // local: Rg - Rl in binades (even, >= 0)
  int extreme;            // weights 2^((z - mg) * c), one frame for all CTAs
  int err;
  int mode;               // RM_*
  int stage;              // ST_*
  int tkind;              // T_*
  int then_mass;          // general path: mass target after the count target
  int nlev;
  float P;
  int kk;                 // top-k size (k' <= V)
  unsigned long long Y;   // mass target: kept iff exclusive mass <= Y
  unsigned long long need;   // count target
  unsigned long long above_m, above_c;
  int ebin;
  uint32_t klo, khi;
  int kshift, nsub;
  float zlo_f, zhi_f;
  unsigned long long Z;   // mass of all tokens
  // result
  float zt;               // cut logit: kept iff z > zt, or z == zt and id <= idcut
  int idcut;              // local: rule for this CTA's ties (INT_MAX all, -1 none)
  int partial;            // local: this CTA must find idcut among its ties
  uint32_t quota;         // local: ties this CTA keeps when partial
  unsigned long long Zk;  // kept mass (fixed 2^-44)
  float invZ;             // 2^44 / Zk
};

struct Shared {
  unsigned long long full[NSMAX];       // slot mbarriers
  X1Row x1[2][2];                       // [exchange parity][row]
  X3 x3;
  RowG rg[2];
  float Rc[2][16];                      // per-CTA frames (cluster copies)
  uint32_t coff[2][17];                 // candidate offsets per CTA
  unsigned long long gb[2][NB];         // merged bins
  uint32_t gc[2][NB];
  unsigned long long scan64[NWARP];
  unsigned long long scan64b[NWARP];
  uint32_t scan32[NWARP];
  float redf[NWARP];
  uint32_t redu[NWARP];
  uint32_t list_n[2];
  int res_i[8];
  unsigned long long res_u[8];
  Meta meta[MR];
  uint32_t timeout;
};

// Dynamic shared memory layout: [Shared][slots][H][G]
//   H (union): per-thread bins float[NB][NT] + counts u8[NB][NT] | top-k lists
//              u64[2][LC] | refinement exchange X2Row[2 parity][2 rows]
//   G (union): per-CTA shifted bins for the merge | gathered candidates u64[GCAP]
//              | per-thread sampling sums
constexpr size_t cmax(size_t a, size_t b) { return a > b ? a : b; }
constexpr size_t H_BYTES = cmax(cmax(4 * sizeof(X2Row), (size_t)NB * NT * 5), 2 * LC * 8);
constexpr size_t G_BYTES = cmax(cmax((size_t)GCAP * 8, (size_t)4 * NT * 8), (size_t)2 * 16 * NB * 12);
constexpr size_t SHARED_BYTES = (sizeof(Shared) + 127) & ~(size_t)127;

#ifdef SV_TRACE
// Phase timestamps of the first 64 units of CTA 0 of cluster 0 (trace builds).
__device__ unsigned long long g_trace[64 * 32 + 16];
#define SV_MARK(k)                                                         \
  do {                                                                     \
    if (cid == 0 && rank == 0 && threadIdx.x == 0 && j < 64)               \
      g_trace[j * 32 + (k)] = global_timer_ns();                           \
  } while (0)
#else
#define SV_MARK(k) \
  do {             \
  } while (0)
#endif

// ------------------------------------------------------------ logit access
// Logits of a slot; keys are 16-bit for bf16 (the logit's full bit pattern in
// order) and 32-bit for fp32.
template <typename DT>
struct Lg;
template <>
struct Lg<__nv_bfloat16> {
  static constexpr int ES = 2;
  __device__ static __forceinline__ float at(const void* s, int l) {
    return __uint_as_float(lds_u16(smem_addr(s) + 2u * (uint32_t)l) << 16);
  }
  __device__ static __forceinline__ uint32_t key(float z) { return okey(z) >> 16; }
  __device__ static __forceinline__ float key_float(uint32_t k) {
    return key_to_float((k << 16) | ((k & 0x8000u) ? 0u : 0xFFFFu));
  }
};
template <>
struct Lg<float> {
  static constexpr int ES = 4;
  __device__ static __forceinline__ float at(const void* s, int l) {
    return __uint_as_float(lds_u32(smem_addr(s) + 4u * (uint32_t)l));
  }
  __device__ static __forceinline__ uint32_t key(float z) { return okey(z); }
  __device__ static __forceinline__ float key_float(uint32_t k) { return key_to_float(k); }
};

__device__ __forceinline__ float to_float_dt(float v) { return v; }
__device__ __forceinline__ float to_float_dt(__nv_bfloat16 v) { return __bfloat162float(v); }

// Calls f(z, l) for every logit of the slot in coalesced 16-byte vectors
// (thread t takes vectors t, t + NT, ...; l is the index in the slice).
template <typename DT, typename F>
__device__ __forceinline__ void for_each_logit(const void* slot, int nvec, F&& f) {
  const uint4* v = reinterpret_cast<const uint4*>(slot);
  for (int q = threadIdx.x; q < nvec; q += NT) {
    const uint4 w = v[q];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    if constexpr (sizeof(DT) == 2) {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        f(__uint_as_float(ws[h] << 16), q * 8 + 2 * h);
        f(__uint_as_float(ws[h] & 0xFFFF0000u), q * 8 + 2 * h + 1);
      }
    } else {
#pragma unroll
      for (int h = 0; h < 4; ++h) f(__uint_as_float(ws[h]), q * 4 + h);
    }
  }
}

// --------------------------------------------------------------- weights
// Bin of a weight e in [0, 2): two binades per bin, the last bin takes the rest.
__device__ __forceinline__ int wbin(float e) {
  return 63 - (int)max(__float_as_uint(e) >> 24, (uint32_t)(64 - NB));
}
// Weight in the CTA frame (normal rows): 2^(z*c - Rl).
__device__ __forceinline__ float wloc(float z, float c, float negR) {
  return ex2_approx(fmaf(z, c, negR));
}
// Weight of rows whose frames cannot be used (|max * c| too large): one frame
// for the cluster, 2^((z - mg) * c).
__device__ __forceinline__ float wext(float z, float mg, float c) {
  return ex2_approx(z == mg ? 0.0f : (z - mg) * c);
}
// Weight of logit z in this CTA's frame (bulk weight).
__device__ __forceinline__ float wbulk(float z, const RowG& g) {
  return g.extreme ? wext(z, g.mg, g.c) : wloc(z, g.c, -g.Rl);
}
// Fixed-point weight in the cluster frame from a CTA-frame weight.
__device__ __forceinline__ unsigned long long fixg(float e, int sh) {
  return fix_pow2(e, FIX - sh);
}
// Bulk weight of logit z as CTA r computes it, in the cluster frame (fixed).
__device__ __forceinline__ unsigned long long fix_of(float z, const RowG& g, float Rr) {
  if (g.extreme) return fixg(wext(z, g.mg, g.c), 0);
  if (!(Rr > -INFINITY)) return 0ull;           // CTA without finite logits
  return fixg(wloc(z, g.c, -Rr), (int)(g.Rg - Rr));
}
// Weight used for probabilities, in the cluster frame: the product z*c is kept
// exactly as a two-term sum and split into integer and fraction, so the
// fraction keeps full precision. It uses the same c as the bulk weights (whose
// sums normalise it), so numerator and normaliser agree to rounding.
__device__ __forceinline__ float wacc(float z, const RowG& g) {
  if (g.extreme) return wext(z, g.mg, g.c);
  const float t = z * g.c;
  if (!(t > -1.0e9f)) return 0.0f;               // -inf logit, or 2^(very negative)
  const float tl = fmaf(z, g.c, -t);
  const float n = rintf(t);
  const float f = (t - n) + tl;
  return ex2_approx(f) * pow2i((int)(n - g.Rg));
}
// The row constants of the sampling phase, passed by value (registers).
struct WP {
  float zt, invZ, c, Rg, mg;
  int idcut, extreme;
};
__device__ __forceinline__ WP wp_of(const RowG& g) {
  WP w;
  w.zt = g.zt;
  w.invZ = g.invZ;
  w.c = g.c;
  w.Rg = g.Rg;
  w.mg = g.mg;
  w.idcut = g.idcut;
  w.extreme = g.extreme;
  return w;
}
__device__ __forceinline__ float wacc_v(float z, WP g) {
  if (g.extreme) return wext(z, g.mg, g.c);
  const float t = z * g.c;
  if (!(t > -1.0e9f)) return 0.0f;
  const float tl = fmaf(z, g.c, -t);
  const float n = rintf(t);
  const float f = (t - n) + tl;
  return ex2_approx(f) * pow2i((int)(n - g.Rg));
}
__device__ __forceinline__ unsigned long long fixr(float p) {
  return fix_pow2(p, 40);
}
__device__ __forceinline__ bool kept(float z, int gid, float zt, int idcut) {
  return z > zt || (z == zt && gid <= idcut);
}

// Exclusive-mass threshold of a top-p cut: a token is kept iff the mass before
// it (fixed point) is <= Y, i.e. < P * Z exactly. P in (0, 1) is m * 2^-s with a
// 24-bit integer m, so Y = floor((m * Z - 1) / 2^s) in 128-bit arithmetic.
__device__ __forceinline__ unsigned long long mass_threshold(float P, unsigned long long Z) {
  int e;
  const float fr = frexpf(P, &e);                 // P = fr * 2^e, fr in [0.5, 1)
  const unsigned long long m = (unsigned long long)(fr * 16777216.0f);
  const int s = 24 - e;                           // >= 24
  unsigned long long lo = m * Z, hi = __umul64hi(m, Z);
  if (lo == 0ull && hi == 0ull) return 0ull;
  if (lo == 0ull) --hi;
  --lo;
  if (s >= 128) return 0ull;
  if (s >= 64) return hi >> (s - 64);
  return (hi << (64 - s)) | (lo >> s);
}

}  // namespace sv
#include "keyhist.cuh"
#include "fstream.cuh"
namespace sv {

// --------------------------------------------------------- block helpers
__device__ __forceinline__ float block_max_nan(float v, float* red) {
  v = warp_max_nan(v);
  __syncthreads();
  if (lane_id() == 0) red[warp_id()] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int i = 1; i < NWARP; ++i) r = fmax_nan(r, red[i]);
  return r;
}
__device__ __forceinline__ uint32_t block_min_u32(uint32_t v, uint32_t* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane_id() == 0) red[warp_id()] = v;
  __syncthreads();
  uint32_t r = red[0];
#pragma unroll
  for (int i = 1; i < NWARP; ++i) r = min(r, red[i]);
  return r;
}

// ------------------------------------------------------------------ passes
// Per-thread maximum of a slot (NaN propagates).
template <typename DT>
__device__ __forceinline__ float thread_max(const void* slot, int nvec) {
  const uint4* v = reinterpret_cast<const uint4*>(slot);
  if constexpr (sizeof(DT) == 2) {
    __nv_bfloat162 m2 = __floats2bfloat162_rn(-INFINITY, -INFINITY);
    for (int q = threadIdx.x; q < nvec; q += NT) {
      const uint4 w = v[q];
      __nv_bfloat162 a, b, c, d;
      memcpy(&a, &w.x, 4);
      memcpy(&b, &w.y, 4);
      memcpy(&c, &w.z, 4);
      memcpy(&d, &w.w, 4);
      m2 = __hmax2_nan(__hmax2_nan(m2, a), __hmax2_nan(__hmax2_nan(b, c), d));
    }
    return fmax_nan(__low2float(m2), __high2float(m2));
  } else {
    float m = -INFINITY;
    for (int q = threadIdx.x; q < nvec; q += NT) {
      const uint4 w = v[q];
      m = fmax_nan(fmax_nan(m, __uint_as_float(w.x)),
                   fmax_nan(__uint_as_float(w.y), fmax_nan(__uint_as_float(w.z), __uint_as_float(w.w))));
    }
    return m;
  }
}

// Lowest slice index holding the value m in this thread's vectors (UINT_MAX if none).
template <typename DT>
__device__ __noinline__ uint32_t thread_first_index(const void* slot, int nvec, float m) {
  const uint4* v = reinterpret_cast<const uint4*>(slot);
  constexpr int PV = 16 / sizeof(DT);
  for (int q = threadIdx.x; q < nvec; q += NT) {
    const uint4 w = v[q];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      if constexpr (sizeof(DT) == 2) {
        if (__uint_as_float(ws[h] << 16) == m) return (uint32_t)(q * PV + 2 * h);
        if (__uint_as_float(ws[h] & 0xFFFF0000u) == m) return (uint32_t)(q * PV + 2 * h + 1);
      } else {
        if (__uint_as_float(ws[h]) == m) return (uint32_t)(q * PV + h);
      }
    }
  }
  return UINT_MAX;
}

// Pass B: per-thread bin masses (and counts) of the slot's weights, then the
// CTA's fixed-point bin masses in the CTA frame, written to x.bins / x.cnts.
template <typename DT, bool COUNTS>
__device__ __noinline__ void pass_bins(const void* slot, int nvec, int vlen, const RowG& g, float* hist,
                          uint8_t* hcnt, X1Row& x) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    hist[j * NT + tid] = 0.0f;
    if (COUNTS) hcnt[j * NT + tid] = 0;
  }
  float* hb = hist + tid + 63 * NT;
  uint8_t* cb = hcnt + tid + 63 * NT;
  if (!g.extreme) {
    const float c = g.c, negR = -g.Rl;
    for_each_logit<DT>(slot, nvec, [&](float z, int l) {
      const float e = wloc(z, c, negR);
      const int o = -(int)max(__float_as_uint(e) >> 24, (uint32_t)(64 - NB)) * NT;
      hb[o] += e;
      if (COUNTS && l < vlen) cb[o] += 1;
    });
  } else {
    const float c = g.c, mg = g.mg;
    for_each_logit<DT>(slot, nvec, [&](float z, int l) {
      const float e = wext(z, mg, c);
      const int o = -(int)max(__float_as_uint(e) >> 24, (uint32_t)(64 - NB)) * NT;
      hb[o] += e;
      if (COUNTS && l < vlen) cb[o] += 1;
    });
  }
  __syncthreads();
  // warp w reduces bins 2w and 2w+1 (the per-thread counts of one bin stay <= 255:
  // a thread holds at most ept logits of a row)
  const int l = lane_id();
  for (int j = 2 * warp_id(); j < 2 * warp_id() + 2; ++j) {
    unsigned long long s = 0;
    uint32_t n = 0;
#pragma unroll
    for (int k = 0; k < NT / 32; ++k) {
      s += fix_pow2(hist[j * NT + l + 32 * k], FIX);
      if (COUNTS) n += hcnt[j * NT + l + 32 * k];
    }
    s = warp_sum(s);
    if (COUNTS) n = warp_sum(n);
    if (l == 0) {
      x.bins[j] = s;
      x.cnts[j] = COUNTS ? n : 0u;
    }
  }
}

// Top-k rows: the 16-bit key prefix of the CTA's k-th largest per-thread maximum
// (k <= NT), by two rounds of 256-bin counting over the thread maxima.
__device__ __noinline__ uint32_t block_kth_prefix16(float tmax, int k, uint32_t* h, uint32_t* res) {
  const int tid = threadIdx.x;
  const uint32_t key = okey(tmax) >> 16;
  uint32_t above = 0, prefix = 0;
  for (int round = 0; round < 2; ++round) {
    h[tid] = 0;
    __syncthreads();
    const bool in = round == 0 || (key >> 8) == prefix;
    if (in) atomicAdd(&h[round == 0 ? (key >> 8) : (key & 0xFFu)], 1u);
    __syncthreads();
    if (warp_id() == 0) {
      // lane l owns digits 255-8l-7 .. 255-8l (descending); find the digit where
      // the count from the top reaches k - above
      const int l = lane_id();
      uint32_t c[8], s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = h[255 - 8 * l - j];
        s += c[j];
      }
      uint32_t incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (l >= o) incl += t;
      }
      uint32_t run = incl - s;
      const uint32_t want = (uint32_t)k - above;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run < want && run + c[j] >= want) {
          res[0] = (uint32_t)(255 - 8 * l - j);
          res[1] = run;
        }
        run += c[j];
      }
    }
    __syncthreads();
    const uint32_t d = res[0];
    above += res[1];
    prefix = round == 0 ? d : ((prefix << 8) | d);
    __syncthreads();
  }
  return prefix;
}

// Top-k rows: lists (okey << 32 | ~id) of the slot's logits >= zt (cap LC).
template <typename DT>
__device__ __noinline__ void pass_list(const void* slot, int nvec, int vlen, float zt, int base,
                          unsigned long long* list, uint32_t* count) {
  for_each_logit<DT>(slot, nvec, [&](float z, int l) {
    const bool pred = z >= zt && l < vlen;
    const uint32_t mk = __ballot_sync(0xffffffffu, pred);
    if (mk) {
      const int lane = lane_id(), leader = __ffs(mk) - 1;
      uint32_t pos = 0;
      if (lane == leader) pos = atomicAdd(count, (uint32_t)__popc(mk));
      pos = __shfl_sync(0xffffffffu, pos, leader) + __popc(mk & ((1u << lane) - 1u));
      if (pred && pos < (uint32_t)LC)
        list[pos] = ((unsigned long long)okey(z) << 32) | (uint32_t)~(uint32_t)(base + l);
    }
  });
}

// One refinement level: counts (and, when a sub-bin spans several keys,
// fixed-point masses) of the slot's logits that lie in the row's key range and
// whose weight falls in the cut bin. Single-key sub-bins (the usual bf16 case,
// where long runs of equal logits make direct atomics contend) are first
// listed as byte-sized sub-bin indices, then counted warp by warp: a warp sorts
// 32 listed indices and adds each run with one atomic. Entries beyond the list
// capacity are counted directly.
template <typename DT>
__device__ __noinline__ void pass_level(const void* slot, int nvec, int vlen, const RowG& gs, X2Row* x,
                           uint8_t* list, uint32_t* list_n, int cap) {
  // row constants in registers (the loop stores to shared memory, which would
  // otherwise force reloads of the shared row state)
  const float lo = gs.zlo_f, hi = gs.zhi_f, c = gs.c, negR = -gs.Rl, mg = gs.mg;
  const bool extreme = gs.extreme != 0;
  const int hsh = gs.sh >> 1, fsh = extreme ? 0 : gs.sh, ebin = gs.ebin, kshift = gs.kshift;
  const uint32_t klo = gs.klo, nsub = (uint32_t)gs.nsub;
  const bool listed = kshift == 0 && nsub <= 255u;
  // per-thread hit buffers (TB entries each, interleaved so that entry r of the
  // 32 lanes of a warp is one 32-byte row); the count stays in a register and
  // no warp-wide operation runs per logit
  constexpr int TB = 32;
  static_assert(NT * TB <= (int)G_BYTES, "hit buffers exceed their region");
  const int tid = threadIdx.x, lane = lane_id();
  uint8_t* tb = list + (size_t)warp_id() * 32 * TB;           // [TB][32] per warp
  uint32_t n = 0;
  (void)list_n;
  (void)cap;
  const uint4* vv = reinterpret_cast<const uint4*>(slot);
  constexpr int PV = 16 / (int)sizeof(DT);
  for (int q = tid; q < nvec; q += NT) {
    const uint4 w4 = vv[q];
    const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int h = 0; h < PV; ++h) {
      float z;
      if constexpr (sizeof(DT) == 2) z = __uint_as_float((h & 1) ? (ws[h >> 1] & 0xFFFF0000u) : (ws[h >> 1] << 16));
      else z = __uint_as_float(ws[h]);
      const int l = q * PV + h;
      if (z >= lo && z <= hi && l < vlen) {
        const float e = extreme ? wext(z, mg, c) : wloc(z, c, negR);
        const int b = extreme ? wbin(e) : min(wbin(e) + hsh, NB - 1);
        if (b == ebin) {
          const uint32_t sub = (Lg<DT>::key(z) - klo) >> kshift;
          if (sub < nsub) {
            if (listed && n < (uint32_t)TB) {
              tb[n * 32 + lane] = (uint8_t)sub;
              ++n;
            } else {
              atomicAdd(&x->cnt[sub], 1u);
              if (kshift > 0) atomicAdd(&x->mass[sub], fixg(e, fsh));
            }
          }
        }
      }
    }
  }
  if (!listed) return;
  // each warp counts its buffers: round r sorts entry r of its 32 lanes and adds
  // each run of equal sub-bins with one atomic
  uint32_t rounds = n;
#pragma unroll
  for (int o = 16; o; o >>= 1) rounds = max(rounds, __shfl_xor_sync(0xffffffffu, rounds, o));
  for (uint32_t r = 0; r < rounds; ++r) {
    uint32_t v = r < n ? tb[r * 32 + lane] : 0xFFu;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
      for (int jj = k >> 1; jj > 0; jj >>= 1) {
        const uint32_t o = __shfl_xor_sync(0xffffffffu, v, jj);
        const bool up = ((lane & k) == 0) == ((lane & jj) == 0);
        v = up ? min(v, o) : max(v, o);
      }
    }
    const uint32_t prev = __shfl_up_sync(0xffffffffu, v, 1);
    const bool start = lane == 0 || prev != v;
    const uint32_t starts = __ballot_sync(0xffffffffu, start);
    if (start && v != 0xFFu) {
      const uint32_t later = starts & ~((2u << lane) - 1u);
      const int next = later ? __ffs(later) - 1 : 32;
      atomicAdd(&x->cnt[v], (uint32_t)(next - lane));
    }
  }
}

// -------------------------------------------------------- cluster merges
// Warp 0 after an exchange barrier: cluster maximum, flags, frames and list
// sizes of row `rho` (lanes 0..C-1 read CTA lane's X1).
__device__ __noinline__ void merge_head(Shared& S, RowG& g, const X1Row* x1p, int rho, int C, uint32_t rank,
                           bool* err, bool* extreme, bool* over, uint32_t* ncand_total) {
  const int l = lane_id();
  float m = -INFINITY, R = -INFINITY;
  uint32_t fl = 0, nc = 0;
  if (l < C) {
    m = ld_peer_f32(&x1p->m, l);
    fl = ld_peer_u32(&x1p->flags, l);
    R = ld_peer_f32(&x1p->R, l);
    nc = ld_peer_u32(&x1p->ncand, l);
  }
  float mg = warp_max_nan(m);
  float Rg = R;
#pragma unroll
  for (int o = 16; o; o >>= 1) Rg = fmaxf(Rg, __shfl_xor_sync(0xffffffffu, Rg, o));
  uint32_t f = fl;
#pragma unroll
  for (int o = 16; o; o >>= 1) f |= __shfl_xor_sync(0xffffffffu, f, o);
  uint32_t incl = nc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (l >= o) incl += t;
  }
  if (l < 16) {
    S.Rc[rho][l] = R;
    S.coff[rho][l + 1] = incl;
  }
  if (l == 0) S.coff[rho][0] = 0;
  *err = isnan(mg) || (f & (F_NAN | F_PINF)) || !(mg > -INFINITY);
  *extreme = (f & F_EXTREME) != 0;
  *over = (f & F_OVER) != 0 || __shfl_sync(0xffffffffu, incl, 31) > (uint32_t)GCAP;
  *ncand_total = __shfl_sync(0xffffffffu, incl, 31);
  if (l == 0) {
    g.mg = mg;
    g.Rg = Rg;
  }
}

// All threads: cluster bins (and counts) of row rho in the cluster frame.
// Thread (r, j) shifts CTA r's bin j into cluster bin min(j + h_r, NB-1); the
// half-warp of CTA r folds the bins that land in the last bin; then thread j
// sums cluster bin j over the CTAs.
__device__ __noinline__ void merge_bins(Shared& S, const X1Row* x1p, int rho, int C, bool extreme,
                           unsigned long long* tmpb, uint32_t* tmpc) {
  const int t = threadIdx.x, r = t >> 4, j = t & 15;
  unsigned long long v = 0;
  uint32_t n = 0;
  int gj = j;
  if (r < C) {
    const float Rr = S.Rc[rho][r];
    const bool live = extreme || Rr > -INFINITY;
    const int sh = extreme ? 0 : (live ? (int)fminf(S.rg[rho].Rg - Rr, 4096.0f) : 4096);
    const unsigned long long b = ld_peer_u64(&x1p->bins[j], r);
    const uint32_t c = ld_peer_u32(&x1p->cnts[j], r);
    if (live) {
      v = sh >= 64 ? 0ull : (b >> sh);
      n = c;
      gj = min(j + (sh >> 1), NB - 1);
    }
  }
  // fold the bins of this CTA that map to the last cluster bin (16-lane groups)
  unsigned long long vl = gj == NB - 1 ? v : 0ull;
  uint32_t nl = gj == NB - 1 ? n : 0u;
#pragma unroll
  for (int o = 8; o; o >>= 1) {
    vl += __shfl_xor_sync(0xffffffffu, vl, o);
    nl += __shfl_xor_sync(0xffffffffu, nl, o);
  }
  tmpb[r * NB + j] = 0ull;
  tmpc[r * NB + j] = 0u;
  __syncthreads();
  if (r < C) {
    if (gj < NB - 1) {
      tmpb[r * NB + gj] = v;
      tmpc[r * NB + gj] = n;
    } else if (j == NB - 1) {
      tmpb[r * NB + NB - 1] = vl;
      tmpc[r * NB + NB - 1] = nl;
    }
  }
  __syncthreads();
  if (t < NB) {
    unsigned long long sum = 0;
    uint32_t cnt = 0;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      sum += tmpb[q * NB + t];
      cnt += tmpc[q * NB + t];
    }
    S.gb[rho][t] = sum;
    S.gc[rho][t] = cnt;
  }
  __syncthreads();
}

// The weight bin a cut lies in, and the key range of that bin (thread 0).
template <typename DT>
__device__ __noinline__ void ebin_pick(Shared& S, RowG& g, int rho) {
  unsigned long long cm = g.above_m, cc = g.above_c;
  int j = 0;
  for (; j < NB - 1; ++j) {
    const bool stop = g.tkind == T_MASS ? (cm + S.gb[rho][j] > g.Y)
                                        : (cc + S.gc[rho][j] >= g.need);
    if (stop) break;
    cm += S.gb[rho][j];
    cc += S.gc[rho][j];
  }
  g.above_m = cm;
  g.above_c = cc;
  g.ebin = j;
  // bin j holds y = z*c - Rg in [-2j-1, -2j+1) (extreme rows: y = (z - mg)*c)
  const float ylo = -2.0f * j - 1.0f, yhi = -2.0f * j + 1.0f;
  float zlo, zhi;
  if (g.extreme) {
    zlo = g.mg + ylo / g.c;
    zhi = g.mg + yhi / g.c;
  } else {
    zlo = (g.Rg + ylo) / g.c;
    zhi = (g.Rg + yhi) / g.c;
  }
  if (j == 0 || !(zhi == zhi)) zhi = INFINITY;
  if (j == NB - 1 || !(zlo == zlo)) zlo = -INFINITY;
  zlo = zlo - fabsf(zlo) * 1.52587890625e-05f - 1e-30f;   // widen by 2^-16 relative
  zhi = zhi + fabsf(zhi) * 1.52587890625e-05f + 1e-30f;
  g.zlo_f = zlo;
  g.zhi_f = zhi;
  g.klo = Lg<DT>::key(zlo);
  g.khi = Lg<DT>::key(zhi);
  const uint32_t span = g.khi - g.klo;
  const int bits = span ? 32 - __clz(span) : 0;
  g.kshift = max(0, bits - 8);
  g.nsub = (int)(span >> g.kshift) + 1;
  g.stage = ST_KEYS;
}

// After a refinement level: merge the sub-bins of row rho, pick the one holding
// the cut; resolve the run of equal logits when a sub-bin is a single key.
template <typename DT>
__device__ __noinline__ void level_pick(Shared& S, RowG& g, int rho, const X2Row* xp, int C, uint32_t rank,
                           unsigned char* Gr) {
  const int t = threadIdx.x;
  const int s = g.nsub - 1 - t;             // thread order = descending keys
  unsigned long long mass = 0;
  uint32_t cnt = 0;
  uint32_t* pc = reinterpret_cast<uint32_t*>(Gr);          // [16] counts of the picked key
  if (s >= 0) {
    // all peers' loads issued together (no dependency between them)
    uint32_t nn[16];
    unsigned long long mm[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      nn[r] = r < C ? ld_peer_u32(&xp->cnt[s], r) : 0u;
      mm[r] = r < C ? ld_peer_u64(&xp->mass[s], r) : 0ull;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      cnt += nn[r];
      mass += mm[r];
    }
  }
  unsigned long long tm;
  const unsigned long long em = block_excl_scan<unsigned long long>(mass, S.scan64, &tm);
  uint32_t tc;
  const uint32_t ec = block_excl_scan<uint32_t>(cnt, S.scan32, &tc);
  if (t == 0) S.res_i[0] = -1;
  __syncthreads();
  if (s >= 0) {
    bool hit;
    if (g.tkind == T_MASS) hit = g.above_m + em <= g.Y && g.above_m + em + mass > g.Y;
    else hit = g.above_c + ec < g.need && g.above_c + ec + cnt >= g.need;
    if (hit) {
      S.res_i[0] = s;
      S.res_u[0] = em;
      S.res_u[1] = ec;
      for (int r = 0; r < 16; ++r) pc[r] = r < C ? ld_peer_u32(&xp->cnt[s], r) : 0u;
    }
  }
  __syncthreads();
  const int sp = S.res_i[0];
  if (sp >= 0 && g.kshift == 0 && warp_id() == 0) {
    // one logit value: split its run of equal logits by token id, CTA by CTA
    // (lane r handles CTA r's members, which follow CTAs 0..r-1 in id order)
    const int l = lane_id();
    const float zk = Lg<DT>::key_float(g.klo + (uint32_t)sp);
    const uint32_t n = l < C ? pc[l] : 0u;
    const unsigned long long E = l < C ? fix_of(zk, g, S.Rc[rho][l]) : 0ull;
    unsigned long long bm = (unsigned long long)n * E;
    unsigned long long bc = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long a = __shfl_up_sync(0xffffffffu, bm, o);
      const unsigned long long c2 = __shfl_up_sync(0xffffffffu, bc, o);
      if (l >= o) {
        bm += a;
        bc += c2;
      }
    }
    const unsigned long long A = g.above_m + S.res_u[0] + bm - (unsigned long long)n * E;
    const unsigned long long before = g.above_c + S.res_u[1] + bc - n;
    uint32_t take;
    if (g.tkind == T_MASS) {
      if (A > g.Y) take = 0;
      else if (E == 0) take = n;
      else {
        const unsigned long long q = (g.Y - A) / E + 1;
        take = q < n ? (uint32_t)q : n;
      }
    } else {
      take = g.need > before ? (uint32_t)min((unsigned long long)n, g.need - before) : 0u;
    }
    const unsigned long long kept_m =
        g.above_m + S.res_u[0] + warp_sum<unsigned long long>((unsigned long long)take * E);
    const uint32_t my_n = __shfl_sync(0xffffffffu, take, (int)rank);
    const uint32_t my_cnt = __shfl_sync(0xffffffffu, n, (int)rank);
    if (l == 0) {
      g.zt = zk;
      g.quota = my_n;
      g.partial = (my_n > 0 && my_n < my_cnt) ? 1 : 0;
      g.idcut = my_n == my_cnt ? INT_MAX : (my_n == 0 ? -1 : 0);
      if (g.tkind == T_COUNT && g.then_mass) {
        // top-k set found (its mass is kept_m); now the top-p cut inside it
        g.Z = kept_m;
        g.Y = mass_threshold(g.P, kept_m);
        g.tkind = T_MASS;
        g.then_mass = 0;
        g.above_m = 0;
        g.above_c = 0;
        g.nlev = 0;
        ebin_pick<DT>(S, g, rho);
      } else {
        g.Zk = kept_m;
        g.stage = ST_DONE;
      }
    }
  } else if (t == 0) {
    if (sp < 0) {
      g.err = 1;                            // no sub-bin holds the cut: inconsistent data
      g.stage = ST_DONE;
    } else if (g.kshift > 0) {
      g.above_m += S.res_u[0];
      g.above_c += S.res_u[1];
      const uint32_t lo = g.klo + ((uint32_t)sp << g.kshift);
      const uint32_t hi = min(g.khi, lo + ((1u << g.kshift) - 1u));
      g.klo = lo;
      g.khi = hi;
      const uint32_t span = hi - lo;
      const int bits = span ? 32 - __clz(span) : 0;
      g.kshift = max(0, bits - 8);
      g.nsub = (int)(span >> g.kshift) + 1;
      g.zlo_f = Lg<DT>::key_float(lo);
      g.zhi_f = Lg<DT>::key_float(hi);
      if (++g.nlev > MAXLEV) {
        g.err = 1;
        g.stage = ST_DONE;
      }
    }
  }
  __syncthreads();
}

// Sorts n composites (okey << 32 | ~id) in descending order (logit desc, id asc).
// n <= NT: rank sort into out; otherwise bitonic in place (out = in).
__device__ __noinline__ unsigned long long* sort_desc(unsigned long long* in, int n, unsigned long long* out) {
  const int t = threadIdx.x;
  if (n <= NT) {
    if (t < n) {
      const unsigned long long v = in[t];
      int rk = 0;
      for (int q = 0; q < n; ++q) rk += in[q] > v;
      out[rk] = v;
    }
    __syncthreads();
    return out;
  }
  int N = 2;
  while (N < n) N <<= 1;
  for (int p = n + t; p < N; p += NT) in[p] = 0ull;
  __syncthreads();
  for (int k = 2; k <= N; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int p = t; p < N; p += NT) {
        const int q = p ^ jj;
        if (q > p) {
          const unsigned long long a = in[p], c = in[q];
          const bool desc = (p & k) == 0;
          if (desc ? a < c : a > c) {
            in[p] = c;
            in[q] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  return in;
}

// Top-k rows: gather the listed candidates of every CTA, sort them, keep the
// first k, then the top-p prefix of those. Sets zt / idcut (global id) / Zk.
template <typename DT>
__device__ __noinline__ void list_select(Shared& S, RowG& g, int rho, const unsigned long long* lists, int C,
                            uint32_t n, int slice, unsigned long long* gbuf) {
  const int t = threadIdx.x;
  for (uint32_t idx = t; idx < n; idx += NT) {
    int r = 0;
    while (r + 1 < C && S.coff[rho][r + 1] <= idx) ++r;
    gbuf[idx] = ld_peer_u64(&lists[rho * LC + (idx - S.coff[rho][r])], r);
  }
  __syncthreads();
  unsigned long long* sorted = sort_desc(gbuf, (int)n, gbuf + 512);
  const int kk = min(g.kk, (int)n);
  unsigned long long E = 0;
  unsigned long long comp = 0;
  if (t < kk) {
    comp = sorted[t];
    const float z = key_to_float((uint32_t)(comp >> 32));
    const int gid = (int)~(uint32_t)comp;
    E = fix_of(z, g, S.Rc[rho][min(gid / slice, C - 1)]);
  }
  unsigned long long tot;
  const unsigned long long ex = block_excl_scan<unsigned long long>(E, S.scan64, &tot);
  unsigned long long Y = ~0ull;
  if (g.P < 1.0f) Y = mass_threshold(g.P, tot);
  const uint32_t keep = (t < kk && ex <= Y) ? 1u : 0u;
  uint32_t nk;
  block_excl_scan<uint32_t>(keep, S.scan32, &nk);
  if (nk == 0) nk = 1;
  if (t == (int)nk - 1) {
    g.zt = key_to_float((uint32_t)(comp >> 32));
    g.idcut = (int)~(uint32_t)comp;
    g.Zk = ex + E;
    g.Z = tot;
    g.partial = 0;
    g.stage = ST_DONE;
  }
  __syncthreads();
}

// ------------------------------------------------------- phase D helpers
// The partial CTA of a run of equal logits finds the id of its quota-th member
// (token-id order): per-thread counts over contiguous id ranges, a block scan,
// then the thread holding that member scans its range.
template <typename DT>
__device__ __noinline__ void tie_pass(Shared& S, RowG& g, const void* slot, int ept, int vlen, int base) {
  const int t = threadIdx.x;
  const int l0 = t * ept, l1 = min(l0 + ept, vlen);
  const float zt = g.zt;
  uint32_t n = 0;
  for (int l = l0; l < l1; ++l) n += Lg<DT>::at(slot, l) == zt;
  uint32_t tot;
  const uint32_t ex = block_excl_scan<uint32_t>(n, S.scan32, &tot);
  if (ex < g.quota && ex + n >= g.quota) {
    uint32_t k = ex;
    for (int l = l0; l < l1; ++l) {
      if (Lg<DT>::at(slot, l) == zt && ++k == g.quota) {
        g.idcut = base + l;
        break;
      }
    }
  }
  __syncthreads();
}

// Sampling weight of slice index l: the residual (p - q)+ (paired units) or p,
// and p itself (both 0 outside the target's kept set).
template <typename DT>
__device__ __forceinline__ void elem_w(const void* s0, const void* s1, bool paired, WP g0, WP g1,
                                       int l, int base, float* r, float* p) {
  const float zp = Lg<DT>::at(s0, l);
  const int gid = base + l;
  *r = 0.0f;
  *p = 0.0f;
  if (kept(zp, gid, g0.zt, g0.idcut)) {
    const float pp = __fmul_rn(wacc_v(zp, g0), g0.invZ);
    float q = 0.0f;
    if (paired) {
      const float zq = Lg<DT>::at(s1, l);
      if (kept(zq, gid, g1.zt, g1.idcut)) q = __fmul_rn(wacc_v(zq, g1), g1.invZ);
    }
    *r = fmaxf(__fsub_rn(pp, q), 0.0f);
    *p = pp;
  }
}

// Residual and target mass over a contiguous id range, as fixed-point sums (2^-40).
template <typename DT>
__device__ __noinline__ void sample_range(const void* s0, const void* s1, bool paired, WP g0,
                                          WP g1, int l0, int l1, int base, unsigned long long* R,
                                          unsigned long long* Pm) {
  unsigned long long ra = 0, pa = 0;
  for (int l = l0; l < l1; ++l) {
    const float zp = Lg<DT>::at(s0, l);
    if (!(zp > g0.zt || (zp == g0.zt && base + l <= g0.idcut))) continue;
    float r, p;
    elem_w<DT>(s0, s1, paired, g0, g1, l, base, &r, &p);
    ra += fixr(r);
    pa += fixr(p);
  }
  *R = ra;
  *Pm = pa;
}

// Warp: the first id in [a0, a1) at which the running sum (from acc) times 2^24
// exceeds kv * S; `useR` selects the residual or p. -1 if none.
template <typename DT>
__device__ __noinline__ int warp_sample_find(const void* s0, const void* s1, bool paired, WP g0,
                                WP g1, int a0, int a1, int base, unsigned long long acc,
                                bool useR, uint32_t kv, unsigned long long S) {
  const int ln = lane_id();
  for (int c0 = a0; c0 < a1; c0 += 32) {
    const int l = c0 + ln;
    unsigned long long w = 0;
    if (l < a1) {
      float r, p;
      elem_w<DT>(s0, s1, paired, g0, g1, l, base, &r, &p);
      w = fixr(useR ? r : p);
    }
    unsigned long long inc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long v = __shfl_up_sync(0xffffffffu, inc, o);
      if (ln >= o) inc += v;
    }
    const bool hit = l < a1 && mul_gt(acc + inc, 1ull << 24, kv, S);
    const uint32_t bal = __ballot_sync(0xffffffffu, hit);
    if (bal) return base + c0 + __ffs(bal) - 1;
    acc += __shfl_sync(0xffffffffu, inc, 31);
  }
  return -1;
}

// Probabilities of a row slice (truncated-probabilities mode).
template <typename DT>
__device__ __noinline__ void write_probs(const void* slot, WP g, int vlen, int base, float* out) {
  for (int l = threadIdx.x; l < vlen; l += NT) {
    const float z = Lg<DT>::at(slot, l);
    out[base + l] = kept(z, base + l, g.zt, g.idcut) ? __fmul_rn(wacc_v(z, g), g.invZ) : 0.0f;
  }
}

// Publishes one unit's result; the last of the K+1 units of sequence b writes
// the sequence's outputs and re-arms the ticket (leaving the workspace zeroed).
__device__ __noinline__ void publish_unit(const Params& P, int unit, int b, int token, bool flag, bool err) {
  P.ws_units[unit] = (unsigned long long)(uint32_t)token | ((unsigned long long)flag << 32) |
                     ((unsigned long long)err << 33);
  __threadfence();
  const unsigned int old = atomicAdd(&P.ws_tickets[b], 1u);
  if (old != (unsigned int)P.K) return;
  __threadfence();
  int nacc = P.K, bad = 0;
  const volatile unsigned long long* u = P.ws_units;
  auto rec = [&](int q) { return u[q < P.K ? (size_t)b * P.K + q : (size_t)P.B * P.K + b]; };
  for (int q = 0; q <= P.K; ++q) {
    const unsigned long long r = rec(q);
    bad |= (int)((r >> 33) & 1ull);
    if (q < P.K && nacc == P.K && !((r >> 32) & 1ull)) nacc = q;
  }
  const int last = (int)(uint32_t)rec(nacc);
  int32_t* ot = P.out_tokens + (size_t)b * (P.K + 1);
  for (int q = 0; q <= P.K; ++q) {
    int v = -1;
    if (!bad) v = q < nacc ? P.dtok[(size_t)b * P.K + q] : (q == nacc ? last : -1);
    ot[q] = v;
  }
  P.out_n[b] = bad ? -1 : nacc;
  for (int q = 0; q <= P.K; ++q)
    P.ws_units[q < P.K ? (size_t)b * P.K + q : (size_t)P.B * P.K + b] = 0ull;
  P.ws_tickets[b] = 0u;
  if (P.fast_split) P.ws_fb[b] = 0u;             // a sequence keyhist_kernel handed back
}

// ------------------------------------------------------------------ kernel
template <int MODE>
__device__ __forceinline__ void decode_unit(const Params& P, int u, int* b, int* i) {
  if (MODE == MODE_VERIFY) {
    const int nb = P.B * P.K;
    if (u < nb) {
      *b = u / P.K;
      *i = u - *b * P.K;
    } else {
      *b = u - nb;
      *i = P.K;
    }
  } else if (MODE == MODE_PROBS) {
    *b = u;
    *i = 0;
  } else {
    *b = u / P.K;
    *i = u - *b * P.K;
  }
}

template <int MODE>
__device__ __forceinline__ bool param_error(const Params& P, const Meta& m, int i) {
  if (!(m.T >= 0.0f) || m.T == INFINITY || !(m.P > 0.0f) || m.k < 0) return true;
  if (MODE == MODE_VERIFY && i < P.K) {
    if (m.d < 0 || m.d >= P.V) return true;
    if (m.T > 0.0f && P.rows1 == nullptr) return true;
  }
  return false;
}

// Rows a unit reads: 0 on a parameter error, 2 for a sampling position i < K.
template <int MODE>
__device__ __forceinline__ int unit_rows(const Params& P, const Meta& m, int i) {
  if (param_error<MODE>(P, m, i)) return 0;
  if (MODE == MODE_VERIFY && P.greedy_split && m.g) return 0;   // greedy path
  if (MODE == MODE_SAMPLE && P.fast_split && m.g) return 0;      // served by keyhist_sample_kernel
  if (MODE == MODE_PROBS && P.fast_split && m.g) return 0;       // served by keyhist_probs_kernel
  if (MODE == MODE_VERIFY && i < P.K && m.T > 0.0f) return 2;
  return 1;
}

template <typename DT, int MODE>
__device__ __forceinline__ const DT* row_src(const Params& P, int b, int i, int which) {
  const DT* r0 = static_cast<const DT*>(P.rows0);
  if (MODE == MODE_VERIFY) {
    if (which == 0) return r0 + ((size_t)b * (P.K + 1) + i) * P.V;
    return static_cast<const DT*>(P.rows1) + ((size_t)b * P.K + i) * P.V;
  }
  if (MODE == MODE_PROBS) return r0 + (size_t)b * P.V;
  return r0 + ((size_t)b * P.K + i) * P.V;
}

// A sequence served by the greedy path: temperature 0 with valid parameters and
// every drafted token in range (any other sequence goes to the cluster kernel,
// which also reports parameter errors).
__device__ __forceinline__ bool greedy_seq(const Params& P, int b) {
  if (!(P.temp[b] == 0.0f) || !(P.topp[b] > 0.0f) || P.topk[b] < 0) return false;
  for (int q = 0; q < P.K; ++q) {
    const int d = P.dtok[(size_t)b * P.K + q];
    if (d < 0 || d >= P.V) return false;
  }
  return true;
}

template <int MODE>
__device__ __noinline__ void load_meta(Shared& S, const Params& P, int cid, int ncl, int nmine, int j0, int cnt) {
  for (int t = threadIdx.x; t < cnt; t += NT) {
    const int j = j0 + t;
    if (j >= nmine) break;
    int b, i;
    decode_unit<MODE>(P, cid + j * ncl, &b, &i);
    Meta m;
    m.T = P.temp[b];
    m.P = P.topp[b];
    m.k = P.topk[b];
    m.d = (MODE == MODE_VERIFY && i < P.K) ? P.dtok[(size_t)b * P.K + i] : 0;
    // sequences served by greedy_kernel or, unless handed back, keyhist_kernel
    m.g = (MODE == MODE_VERIFY && P.greedy_split)
              ? (int)(greedy_seq(P, b) || (P.fast_split && fast_seq(P, b) && P.ws_fb[b] == 0u))
              : 0;
    // draft sampler: rows keyhist_sample_kernel served (not marked for this kernel)
    if (MODE == MODE_SAMPLE && P.fast_split) m.g = P.out_tokens[(size_t)b * P.K + i] != KH_HANDBACK;
    // truncated probabilities: rows keyhist_probs_kernel wrote (not marked for this kernel)
    if (MODE == MODE_PROBS && P.fast_split)
      m.g = __float_as_uint(P.out_probs[(size_t)b * P.V]) != KH_PROBS_HANDBACK;
    S.meta[j % MR] = m;
  }
}

template <typename DT>
__device__ __forceinline__ DT neg_inf();
template <>
__device__ __forceinline__ float neg_inf<float>() {
  return -INFINITY;
}
template <>
__device__ __forceinline__ __nv_bfloat16 neg_inf<__nv_bfloat16>() {
  return __ushort_as_bfloat16((unsigned short)0xFF80u);
}

template <typename DT, int MODE>
__global__ void __launch_bounds__(NT, 2) sv_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem[];
  Shared& S = *reinterpret_cast<Shared*>(smem);
  const size_t slot_bytes = (size_t)P.slot_elems * sizeof(DT);
  unsigned char* slots = smem + SHARED_BYTES;
  unsigned char* H = slots + (size_t)P.NS * slot_bytes;
  float* hist = reinterpret_cast<float*>(H);
  uint8_t* hcnt = H + (size_t)NB * NT * 4;
  unsigned long long* lists = reinterpret_cast<unsigned long long*>(H);
  X2Row* x2 = reinterpret_cast<X2Row*>(H);
  unsigned char* Gr = H + H_BYTES;
  unsigned long long* gbuf = reinterpret_cast<unsigned long long*>(Gr);

  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank();
  const int C = P.C;
  const int cid = (int)cluster_id_x(), ncl = (int)num_clusters_x();
  const int base = (int)rank * P.slice;
  const int vlen = max(0, min(P.slice, P.V - base));
  const int nvec = (int)(slot_bytes / 16);
  // launched early (programmatic dependent launch) behind greedy_kernel and
  // keyhist_kernel: wait until they are done before reading what they wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int nmine = cid < P.nunits ? (P.nunits - 1 - cid) / ncl + 1 : 0;
  // verify batches whose units are all served by greedy_kernel or keyhist_kernel:
  // nothing to do here (every CTA reads the same flag, so none waits on another)
  if (MODE == MODE_VERIFY && P.greedy_split && *reinterpret_cast<volatile unsigned int*>(P.ws_work) == 0u)
    return;
  // draft sampler: nothing left when no row carries the hand-back mark (every CTA
  // scans the same outputs, so all of a cluster decide alike)
  if (MODE == MODE_SAMPLE && P.fast_split && P.nunits <= 65536) {
    int marked = 0;
    for (int t = threadIdx.x; t < P.nunits; t += NT) marked |= P.out_tokens[t] == KH_HANDBACK;
    if (!__syncthreads_or(marked)) return;
  }
  const uint32_t copy_bytes = (uint32_t)((size_t)vlen * sizeof(DT));
  const uint64_t pol = policy_evict_first();

  if (tid == 0) {
    for (int s = 0; s < P.NS; ++s) mbar_init(&S.full[s], 1);
    fence_mbar_init();
    S.timeout = 0;
  }
  for (int s = 0; s < P.NS; ++s) {
    DT* sp = reinterpret_cast<DT*>(slots + (size_t)s * slot_bytes);
    for (int l = vlen + tid; l < P.slot_elems; l += NT) sp[l] = neg_inf<DT>();
  }
  load_meta<MODE>(S, P, cid, ncl, nmine, 0, MR);
  __syncthreads();

  int next_j = 0, rows_issued = 0, rows_done = 0, xr = 0, lp = 0;

  for (int j = 0; j < nmine; ++j) {
    if (j > 0 && (j % (MR / 2)) == 0) {
      __syncthreads();
      load_meta<MODE>(S, P, cid, ncl, nmine, j + MR / 2, MR / 2);
      __syncthreads();
    }
    // producer: row slices of the next units, as far as the slots allow
    if (P.bulk_ok && !S.timeout) {
      bool fenced = false;
      // only units whose metadata is loaded (the ring holds units j .. j+MR/2-1
      // at least)
      const int jlim = min(nmine, j + MR / 2);
      while (next_j < jlim) {
        int nb_, ni_;
        decode_unit<MODE>(P, cid + next_j * ncl, &nb_, &ni_);
        const int nr = unit_rows<MODE>(P, S.meta[next_j % MR], ni_);
        if (rows_issued - rows_done + nr > P.NS) break;
        if (tid == 0) {
          if (!fenced) {
            fence_proxy_async();
            fenced = true;
          }
          for (int w = 0; w < nr; ++w) {
            const int s = (rows_issued + w) % P.NS;
            mbar_arrive_expect_tx(&S.full[s], copy_bytes);
            if (copy_bytes)
              bulk_g2s(slots + (size_t)s * slot_bytes, row_src<DT, MODE>(P, nb_, ni_, w) + base,
                       copy_bytes, &S.full[s], pol);
          }
        }
        rows_issued += nr;
        ++next_j;
      }
    }
    const int u = cid + j * ncl;
    int b, i;
    decode_unit<MODE>(P, u, &b, &i);
    const Meta m = S.meta[j % MR];
    SV_MARK(0);
    const bool perr = param_error<MODE>(P, m, i);
    const int nr = unit_rows<MODE>(P, m, i);
    const void* sl[2] = {slots + (size_t)(rows_done % P.NS) * slot_bytes,
                         slots + (size_t)((rows_done + 1) % P.NS) * slot_bytes};
    // consumer: wait for (or, without bulk copies, load) the unit's rows
    if (P.bulk_ok) {
      if (!S.timeout) {
        for (int w = 0; w < nr; ++w) {
          const int ri = rows_done + w;
          if (!mbar_wait_bounded(&S.full[ri % P.NS], (uint32_t)((ri / P.NS) & 1), WAIT_LIMIT_NS)) {
            atomicOr(&S.timeout, 1u);
            atomicOr(P.ws_error, 1u);
          }
        }
      }
    } else {
      for (int w = 0; w < nr; ++w) {
        DT* dst = reinterpret_cast<DT*>(const_cast<void*>(sl[w]));
        const DT* src = row_src<DT, MODE>(P, b, i, w) + base;
        for (int l = tid; l < vlen; l += NT) dst[l] = src[l];
      }
    }
    __syncthreads();
    const bool tmo = S.timeout != 0;
    SV_MARK(1);

    if (perr) {
      // ------------------------------------------------ parameter error
      if (MODE == MODE_VERIFY) {
        if (rank == 0 && tid == 0) publish_unit(P, u, b, -1, false, true);
      } else if (MODE == MODE_SAMPLE) {
        if (rank == 0 && tid == 0) P.out_tokens[(size_t)b * P.K + i] = -1;
      } else {
        for (int l = tid; l < vlen; l += NT) P.out_probs[(size_t)b * P.V + base + l] = __int_as_float(0x7fc00000);
      }
    } else if ((MODE == MODE_VERIFY && P.greedy_split && m.g) ||
               ((MODE == MODE_SAMPLE || MODE == MODE_PROBS) && P.fast_split && m.g)) {
      // units served by greedy_kernel, keyhist_kernel, keyhist_sample_kernel or
      // keyhist_probs_kernel
    } else if (m.T == 0.0f) {
      // ------------------------------------------------ greedy (T = 0)
      X1Row& x = S.x1[xr & 1][0];
      const float tm = thread_max<DT>(sl[0], nvec);
      const float mx = block_max_nan(tm, S.redf);
      uint32_t fi = UINT_MAX;
      if (mx > -INFINITY && mx < INFINITY) fi = thread_first_index<DT>(sl[0], nvec, mx);
      fi = block_min_u32(fi, S.redu);
      if (tid == 0) {
        x.m = mx;
        x.flags = ((isnan(mx) || tmo) ? F_NAN : 0u) | (mx == INFINITY ? F_PINF : 0u);
        x.best = (fi < (uint32_t)vlen) ? (((unsigned long long)okey(mx) << 32) | (uint32_t)~(uint32_t)(base + (int)fi)) : 0ull;
      }
      cluster_sync();
      if (warp_id() == 0) {
        const int l = lane_id();
        unsigned long long bst = 0;
        uint32_t fl = 0;
        float mm = -INFINITY;
        if (l < C) {
          bst = ld_peer_u64(&x.best, l);
          fl = ld_peer_u32(&x.flags, l);
          mm = ld_peer_f32(&x.m, l);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const unsigned long long ob = __shfl_xor_sync(0xffffffffu, bst, o);
          bst = ob > bst ? ob : bst;
          fl |= __shfl_xor_sync(0xffffffffu, fl, o);
        }
        mm = warp_max_nan(mm);
        if (l == 0) {
          S.res_i[0] = (fl & (F_NAN | F_PINF)) || !(mm > -INFINITY) || bst == 0ull;
          S.res_i[1] = (int)~(uint32_t)bst;
        }
      }
      __syncthreads();
      const bool err = S.res_i[0] != 0;
      const int amax = S.res_i[1];
      if (MODE == MODE_VERIFY) {
        if (rank == 0 && tid == 0) publish_unit(P, u, b, err ? -1 : amax, i < P.K && m.d == amax, err);
      } else if (MODE == MODE_SAMPLE) {
        if (rank == 0 && tid == 0) P.out_tokens[(size_t)b * P.K + i] = err ? -1 : amax;
      } else {
        for (int l = tid; l < vlen; l += NT)
          P.out_probs[(size_t)b * P.V + base + l] =
              err ? __int_as_float(0x7fc00000) : (base + l == amax ? 1.0f : 0.0f);
      }
      ++xr;
    } else {
      // ------------------------------------------------ sampling unit
      const bool paired = nr == 2;
      if (tid == 0) {
        for (int rho = 0; rho < nr; ++rho) {
          RowG& g = S.rg[rho];
          g = RowG{};
          g.c = __fdiv_rn(1.44269504088896341f, m.T);   // log2(e)/T
          g.P = m.P;
          const int kk = (m.k > 0 && m.k < P.V) ? m.k : P.V;
          g.kk = kk;
          g.mode = kk < P.V ? (kk <= KFAST ? RM_LIST : RM_GENERAL) : (m.P < 1.0f ? RM_TOPP : RM_ALL);
          g.zt = -INFINITY;
          g.idcut = INT_MAX;
          g.Rl = -INFINITY;
        }
      }
      __syncthreads();
      // pass A and pass B (or the top-k candidate list) of each row
      X1Row* X = S.x1[xr & 1];
      for (int rho = 0; rho < nr; ++rho) {
        RowG& g = S.rg[rho];
        const float tm = thread_max<DT>(sl[rho], nvec);
        const float mx = block_max_nan(tm, S.redf);
        const bool fin = mx > -INFINITY && mx < INFINITY;
        bool ext = false;
        float R = -INFINITY;
        if (fin) {
          const float mc = mx * g.c;
          if (!(fabsf(mc) < 4194304.0f)) ext = true;
          else R = 2.0f * ceilf(mc * 0.5f);
        }
        if (tid == 0) {
          X[rho].m = mx;
          X[rho].flags = ((isnan(mx) || tmo) ? F_NAN : 0u) | (mx == INFINITY ? F_PINF : 0u) |
                         (ext ? F_EXTREME : 0u);
          X[rho].R = R;
          X[rho].ncand = 0;
          g.Rl = R;
          S.list_n[rho] = 0;
        }
        if (tid < NB) {
          X[rho].bins[tid] = 0ull;
          X[rho].cnts[tid] = 0u;
        }
        __syncthreads();
        if (g.mode == RM_LIST) {
          if (fin) {
            const uint32_t t16 = block_kth_prefix16(tm, g.kk, reinterpret_cast<uint32_t*>(Gr),
                                                    reinterpret_cast<uint32_t*>(S.res_i));
            const float zt = t16 <= 0x007Fu ? -INFINITY : key_to_float(t16 << 16);
            pass_list<DT>(sl[rho], nvec, vlen, zt, base, lists + rho * LC, &S.list_n[rho]);
            __syncthreads();
            if (tid == 0) {
              X[rho].ncand = min(S.list_n[rho], (uint32_t)LC);
              if (S.list_n[rho] > (uint32_t)LC) X[rho].flags |= F_OVER;
            }
          }
        } else if (fin && !ext) {
          if (g.mode == RM_GENERAL) pass_bins<DT, true>(sl[rho], nvec, vlen, g, hist, hcnt, X[rho]);
          else pass_bins<DT, false>(sl[rho], nvec, vlen, g, hist, hcnt, X[rho]);
        }
        __syncthreads();
        if (rho == 0) SV_MARK(11);
      }
      SV_MARK(2);
      cluster_sync();                                              // S1
      SV_MARK(3);
      // cluster maxima, frames, flags
      if (warp_id() == 0) {
        for (int rho = 0; rho < nr; ++rho) {
          bool e, ex, ov;
          uint32_t ntot;
          merge_head(S, S.rg[rho], &X[rho], rho, C, rank, &e, &ex, &ov, &ntot);
          if (lane_id() == 0) {
            RowG& g = S.rg[rho];
            g.err = e;
            g.extreme = ex;
            g.sh = ex ? 0 : (g.Rl > -INFINITY ? (int)fminf(g.Rg - g.Rl, 4096.0f) : 4096);
            S.res_i[2 + rho] = ov ? -1 : (int)ntot;
          }
        }
      }
      __syncthreads();
      SV_MARK(22);
      ++xr;
      bool uerr = S.rg[0].err || (paired && S.rg[1].err);
      if (!uerr) {
        // rows that need bins: merge them; rows whose bins must be (re)computed
        // in the cluster frame (extreme) or with counts (overflowing lists) get
        // one more exchange round
        // (both rows of a unit share their parameters, so both list or neither;
        // if either list overflowed, both rows take the general path and no CTA
        // reads another's lists)
        const bool lists_over = S.rg[0].mode == RM_LIST &&
                                (S.res_i[2] < 0 || (paired && S.res_i[3] < 0));
        bool redo = false;
        for (int rho = 0; rho < nr; ++rho) {
          RowG& g = S.rg[rho];
          const bool was_list = g.mode == RM_LIST;
          __syncthreads();
          if (tid == 0) S.res_i[2 + rho] = (was_list && lists_over) ? -1 : S.res_i[2 + rho];
          if (tid == 0 && was_list && lists_over) g.mode = RM_GENERAL;
          __syncthreads();
          if (g.mode == RM_LIST) continue;
          if (g.extreme || (was_list && lists_over)) redo = true;
          else merge_bins(S, &X[rho], rho, C, false, gbuf, reinterpret_cast<uint32_t*>(gbuf + 16 * NB));
        }
        if (redo) {
          X1Row* X2_ = S.x1[xr & 1];
          for (int rho = 0; rho < nr; ++rho) {
            RowG& g = S.rg[rho];
            const bool need = g.mode != RM_LIST && (g.extreme || S.res_i[2 + rho] < 0);
            if (tid < NB) {
              X2_[rho].bins[tid] = 0ull;
              X2_[rho].cnts[tid] = 0u;
            }
            if (tid == 0) {
              X2_[rho].m = g.mg;
              X2_[rho].flags = 0;
              X2_[rho].R = g.Rl;
              X2_[rho].ncand = 0;
            }
            __syncthreads();
            if (need && (g.extreme || g.Rl > -INFINITY)) {
              if (g.mode == RM_GENERAL) pass_bins<DT, true>(sl[rho], nvec, vlen, g, hist, hcnt, X2_[rho]);
              else pass_bins<DT, false>(sl[rho], nvec, vlen, g, hist, hcnt, X2_[rho]);
            }
            __syncthreads();
          }
          cluster_sync();                                          // S1b
          for (int rho = 0; rho < nr; ++rho) {
            RowG& g = S.rg[rho];
            const bool need = g.mode != RM_LIST && (g.extreme || S.res_i[2 + rho] < 0);
            if (need)
              merge_bins(S, &X2_[rho], rho, C, g.extreme != 0, gbuf,
                         reinterpret_cast<uint32_t*>(gbuf + 16 * NB));
          }
          ++xr;
        }
        SV_MARK(23);
        // selection set-up
        for (int rho = 0; rho < nr; ++rho) {
          RowG& g = S.rg[rho];
          if (g.mode == RM_LIST) {
            list_select<DT>(S, g, rho, lists, C, (uint32_t)S.res_i[2 + rho], P.slice, gbuf);
            continue;
          }
          if (tid == 0) {
            unsigned long long Z = 0;
            for (int q = 0; q < NB; ++q) Z += S.gb[rho][q];
            g.Z = Z;
            if (g.mode == RM_ALL) {
              g.zt = -INFINITY;
              g.idcut = INT_MAX;
              g.Zk = Z;
              g.stage = ST_DONE;
            } else if (g.mode == RM_TOPP) {
              g.tkind = T_MASS;
              g.Y = mass_threshold(g.P, Z);
              ebin_pick<DT>(S, g, rho);
            } else {
              g.tkind = T_COUNT;
              g.need = (unsigned long long)g.kk;
              g.then_mass = g.P < 1.0f;
              ebin_pick<DT>(S, g, rho);
            }
          }
          __syncthreads();
        }
        SV_MARK(4);
        // refinement levels (one cluster barrier each)
        while (true) {
          const bool k0 = S.rg[0].stage == ST_KEYS && !S.rg[0].err;
          const bool k1 = paired && S.rg[1].stage == ST_KEYS && !S.rg[1].err;
          if (!k0 && !k1) break;
          X2Row* xl = x2 + (lp & 1) * 2;
          for (int rho = 0; rho < nr; ++rho) {
            if (rho == 0 ? !k0 : !k1) continue;
            for (int q = tid; q < NSUB; q += NT) {
              xl[rho].cnt[q] = 0u;
              xl[rho].mass[q] = 0ull;
            }
          }
          if (tid < 2) S.list_n[tid] = 0u;
          __syncthreads();
          SV_MARK(16);
          for (int rho = 0; rho < nr; ++rho) {
            if (rho == 0 ? !k0 : !k1) continue;
            // the hit buffers (8 KB) are consumed inside the call, so rows share them
            pass_level<DT>(sl[rho], nvec, vlen, S.rg[rho], &xl[rho], Gr, &S.list_n[rho], (int)G_BYTES);
            SV_MARK(17 + rho);
          }
          __syncthreads();
          SV_MARK(19);
          // single-key sub-bins: mass = count * this CTA's weight of that key
          for (int rho = 0; rho < nr; ++rho) {
            if (rho == 0 ? !k0 : !k1) continue;
            const RowG& g = S.rg[rho];
            if (g.kshift == 0 && tid < g.nsub) {
              const uint32_t n = xl[rho].cnt[tid];
              if (n) {
                const float zk = Lg<DT>::key_float(g.klo + (uint32_t)tid);
                xl[rho].mass[tid] = (unsigned long long)n * fix_of(zk, g, g.Rl);
              }
            }
          }
          SV_MARK(13);
          cluster_sync();                                          // S2 (per level)
          SV_MARK(14);
          for (int rho = 0; rho < nr; ++rho) {
            if (rho == 0 ? !k0 : !k1) continue;
            level_pick<DT>(S, S.rg[rho], rho, &xl[rho], C, rank, Gr);
            SV_MARK(20 + rho);
          }
          ++lp;
#ifdef SV_TRACE
          if (cid == 0 && rank == 0 && threadIdx.x == 0 && j < 64) g_trace[j * 32 + 10] = (unsigned long long)lp;
#endif
        }
        uerr = S.rg[0].err || (paired && S.rg[1].err);
        SV_MARK(5);
      }
      if (uerr) {
        if (MODE == MODE_VERIFY) {
          if (rank == 0 && tid == 0) publish_unit(P, u, b, -1, false, true);
        } else if (MODE == MODE_SAMPLE) {
          if (rank == 0 && tid == 0) P.out_tokens[(size_t)b * P.K + i] = -1;
        } else {
          for (int l = tid; l < vlen; l += NT) P.out_probs[(size_t)b * P.V + base + l] = __int_as_float(0x7fc00000);
        }
        cluster_sync();                                            // end of unit
      } else {
        // ---------------------------------------------- phase D
        if (tid == 0) {
          for (int rho = 0; rho < nr; ++rho) {
            RowG& g = S.rg[rho];
            g.invZ = __fdiv_rn(17592186044416.0f, (float)(g.Zk ? g.Zk : 1ull));   // 2^44 / Zk
          }
        }
        __syncthreads();
        for (int rho = 0; rho < nr; ++rho)
          if (S.rg[rho].partial) tie_pass<DT>(S, S.rg[rho], sl[rho], P.ept, vlen, base);
        __syncthreads();
        SV_MARK(12);
        const WP g0 = wp_of(S.rg[0]);
        const WP g1 = wp_of(S.rg[paired ? 1 : 0]);
        if (MODE == MODE_PROBS) {
          write_probs<DT>(sl[0], g0, vlen, base, P.out_probs + (size_t)b * P.V);
          cluster_sync();                                          // end of unit
        } else {
          uint32_t ku, kv;
          philox_uniform_bits(P.seed, philox_offset_of(P), (uint32_t)b, (uint32_t)i, &ku, &kv);
          if (tid == 0) {
            uint32_t flag = 0;
            if (paired && m.d / P.slice == (int)rank) {
              const int l = m.d - base;
              const float zp = Lg<DT>::at(sl[0], l), zq = Lg<DT>::at(sl[1], l);
              const float p = kept(zp, m.d, g0.zt, g0.idcut) ? __fmul_rn(wacc_v(zp, g0), g0.invZ) : 0.0f;
              const float q = kept(zq, m.d, g1.zt, g1.idcut) ? __fmul_rn(wacc_v(zq, g1), g1.invZ) : 0.0f;
              flag = __fmul_rn((float)ku * 5.9604644775390625e-08f, q) < p ? 1u : 0u;
            }
            S.x3.flag = flag;
          }
          const int l0 = min(tid * P.ept, vlen), l1 = min(l0 + P.ept, vlen);
          unsigned long long Rt, Pt;
          sample_range<DT>(sl[0], sl[1], paired, g0, g1, l0, l1, base, &Rt, &Pt);
          __syncthreads();
          SV_MARK(15);
          unsigned long long totR, totP;
          const unsigned long long exR = block_excl_scan<unsigned long long>(Rt, S.scan64, &totR);
          const unsigned long long exP = block_excl_scan<unsigned long long>(Pt, S.scan64b, &totP);
          if (tid == 0) {
            S.x3.R = totR;
            S.x3.P = totP;
          }
          SV_MARK(6);
          cluster_sync();                                          // S3
          SV_MARK(7);
          if (warp_id() == 0) {
            const int l = lane_id();
            unsigned long long r = 0, p = 0;
            if (l < C) {
              r = ld_peer_u64(&S.x3.R, l);
              p = ld_peer_u64(&S.x3.P, l);
            }
            unsigned long long ir = r, ip = p;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const unsigned long long a = __shfl_up_sync(0xffffffffu, ir, o);
              const unsigned long long c2 = __shfl_up_sync(0xffffffffu, ip, o);
              if (l >= o) {
                ir += a;
                ip += c2;
              }
            }
            const unsigned long long SR = __shfl_sync(0xffffffffu, ir, 31);
            const unsigned long long SP = __shfl_sync(0xffffffffu, ip, 31);
            const bool useR = SR > 0ull;
            const unsigned long long Stot = useR ? SR : SP;
            const unsigned long long inc = useR ? ir : ip, own = useR ? r : p;
            const bool cross = l < C && mul_gt(inc, 1ull << 24, kv, Stot) &&
                               !mul_gt(inc - own, 1ull << 24, kv, Stot);
            const uint32_t bal = __ballot_sync(0xffffffffu, cross);
            const int cs = bal ? __ffs(bal) - 1 : C - 1;
            if (l == cs) {
              S.res_i[4] = cs;
              S.res_i[5] = useR;
              S.res_i[6] = bal ? 1 : 0;
              S.res_u[0] = inc - own;
              S.res_u[1] = Stot;
            }
          }
          __syncthreads();
          if (S.res_i[4] == (int)rank) {
            const bool useR = S.res_i[5] != 0;
            const unsigned long long Stot = S.res_u[1];
            const unsigned long long ex = S.res_u[0] + (useR ? exR : exP);
            const unsigned long long own = useR ? Rt : Pt;
            const bool mine = S.res_i[6] && mul_gt(ex + own, 1ull << 24, kv, Stot) &&
                              !mul_gt(ex, 1ull << 24, kv, Stot);
            if (tid == 0) S.res_i[7] = -1;
            __syncthreads();
            if (mine) {
              S.res_i[7] = tid;
              S.res_u[2] = ex;
            }
            __syncthreads();
            const int ts = S.res_i[7];
            if (warp_id() == 0) {
              int tok = -1;
              if (ts >= 0) {
                const int a0 = min(ts * P.ept, vlen), a1 = min(a0 + P.ept, vlen);
                tok = warp_sample_find<DT>(sl[0], sl[1], paired, g0, g1, a0, a1, base, S.res_u[2],
                                           useR, kv, Stot);
              }
              if (tid == 0) {
                if (MODE == MODE_VERIFY) {
                  bool flag = false;
                  if (paired) flag = ld_peer_u32(&S.x3.flag, (uint32_t)(m.d / P.slice)) != 0u;
                  publish_unit(P, u, b, tok, flag, tok < 0);
                } else {
                  P.out_tokens[(size_t)b * P.K + i] = tok;
                }
              }
            }
          }
          // X3 is read by peers until their next cluster barrier; it is written
          // again only after the next unit's first barrier
        }
      }
    }
    __syncthreads();
    rows_done += nr;
    SV_MARK(8);
#ifdef SV_TRACE
    if (cid == 0 && rank == 0 && threadIdx.x == 0 && j < 64) g_trace[j * 32 + 9] = (unsigned long long)nr;
#endif
  }
#ifdef SV_TRACE
  if (cid == 0 && rank == 0 && threadIdx.x == 0) {
    g_trace[64 * 32] = (unsigned long long)ncl;
    g_trace[64 * 32 + 1] = (unsigned long long)nmine;
  }
#endif
  // copies still in flight after a timeout: wait (bounded) before leaving
  if (tid == 0 && S.timeout && P.bulk_ok) {
    for (int s = 0; s < P.NS && s < rows_issued; ++s) {
      const int last = s + ((rows_issued - 1 - s) / P.NS) * P.NS;   // last fill of slot s
      mbar_wait_bounded(&S.full[s], (uint32_t)((last / P.NS) & 1), WAIT_LIMIT_NS);
    }
  }
  __syncthreads();
  cluster_sync();   // no CTA leaves while another may still read its shared memory
  if (MODE == MODE_VERIFY && tid == 0) {
    // the last CTA to finish re-arms the work flag for the next call (every CTA
    // read it at its start)
    __threadfence();
    if (atomicAdd(P.ws_done, 1u) == gridDim.x - 1u) {
      *P.ws_work = 0u;
      *P.ws_done = 0u;
      // a timed-out wait of this call was already reported in band (its sequences
      // are data errors); clear its flag so the workspace is zero for the next call
      *P.ws_error = 0u;
    }
  }
}

// ------------------------------------------------------- greedy streaming
// Temperature-0 sequences of spec_verify: each target row is split into G chunks
// (items). A persistent grid walks the items; a CTA holds its next item's
// 16-byte vector loads in registers while it reduces the current one, so HBM
// reads stay in flight. Per item: the maximum (packed bf16x2) and the lowest
// index holding it, merged into the row's slot as (okey(max) << 32 | ~index)
// with a 64-bit atomicMax that needs no reply (the largest logit, then the
// lowest id); NaN / +inf set the row's flag. The last CTA to finish writes the
// sequences' outputs. Items of other sequences raise the cluster kernel's work
// flag.
constexpr int GV = 4;          // 16-byte vectors per thread and wave
constexpr int GW = 6;          // waves per item (at most)

// A greedy sequence once all its rows are reduced: the accepted prefix and the
// token from the K+1 rows' (max, argmax) slots, which are cleared for the next call.
__device__ void greedy_finalize_seq(const Params& P, int b, unsigned long long* best,
                                    unsigned int* rflag) {
  const int K = P.K;
  int nacc = K, last = -1;
  bool err = false;
  for (int q = 0; q <= K; ++q) {
    const size_t r = (size_t)b * (K + 1) + q;
    const unsigned long long fb = best[r];
    const unsigned int ff = rflag[r];
    best[r] = 0ull;
    rflag[r] = 0u;
    err |= ff != 0u || fb == 0ull;
    const int amax = (int)~(uint32_t)fb;
    if (nacc == K) {
      if (q < K && P.dtok[(size_t)b * K + q] != amax) {
        nacc = q;
        last = amax;
      } else if (q == K) {
        last = amax;
      }
    }
  }
  int32_t* ot = P.out_tokens + (size_t)b * (K + 1);
  for (int q = 0; q <= K; ++q)
    ot[q] = err ? -1 : (q < nacc ? P.dtok[(size_t)b * K + q] : (q == nacc ? last : -1));
  P.out_n[b] = err ? -1 : nacc;
}

// Geometry of greedy item `item` (row chunk): its row, whether the row belongs
// to a temperature-0 sequence, its first vector and its vector count (0 for rows
// of other sequences, which are not read here).
template <typename DT>
__device__ __forceinline__ void greedy_item(const Params& P, int item, int G, int chunk, int* row_out,
                                            bool* ok_out, const uint4** v_out, int* nv_out, int* l0_out) {
  constexpr int PV = 16 / (int)sizeof(DT);
  const int row = item / G, c = item - row * G;
  const bool ok = greedy_seq(P, row / (P.K + 1));
  const int l0 = c * chunk, l1 = min(l0 + chunk, P.V);
  *row_out = row;
  *ok_out = ok;
  *v_out = reinterpret_cast<const uint4*>(static_cast<const DT*>(P.rows0) + (size_t)row * P.V) + l0 / PV;
  *nv_out = ok ? (l1 - l0) / PV : 0;
  *l0_out = l0;
}
// One wave of an item: vectors w0 + tid + q NT (q < GV), -inf past the chunk.
template <typename DT>
__device__ __forceinline__ void greedy_wave(const uint4* v, int nv, int w0, uint4* x) {
  constexpr uint32_t NEG = sizeof(DT) == 2 ? 0xFF80FF80u : 0xFF800000u;
#pragma unroll
  for (int q = 0; q < GV; ++q) {
    const int vi = w0 + (int)threadIdx.x + q * NT;
    if (vi < nv) {
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(x[q].x), "=r"(x[q].y), "=r"(x[q].z), "=r"(x[q].w)
                   : "l"(v + vi));
    } else {
      x[q] = make_uint4(NEG, NEG, NEG, NEG);
    }
  }
}
// Maximum of one 16-byte vector (NaN if it holds one).
template <typename DT>
__device__ __forceinline__ float greedy_vmax(const uint4& x) {
  if constexpr (sizeof(DT) == 2) {
    __nv_bfloat162 a, bb, cc, dd;
    memcpy(&a, &x.x, 4);
    memcpy(&bb, &x.y, 4);
    memcpy(&cc, &x.z, 4);
    memcpy(&dd, &x.w, 4);
    const __nv_bfloat162 v2 = __hmax2_nan(__hmax2_nan(a, bb), __hmax2_nan(cc, dd));
    return fmax_nan(__low2float(v2), __high2float(v2));
  } else {
    return fmax_nan(fmax_nan(__uint_as_float(x.x), __uint_as_float(x.y)),
                    fmax_nan(__uint_as_float(x.z), __uint_as_float(x.w)));
  }
}

template <typename DT>
__global__ void __launch_bounds__(NT) greedy_kernel(const Params P, int G, int chunk, int nitems,
                                                     unsigned long long* best,
                                                     unsigned int* rflag, unsigned int* done) {
  const int tid = threadIdx.x;
  constexpr int PV = 16 / (int)sizeof(DT);
  constexpr int WV = GV * NT;                  // vectors per wave
  uint4 cur[GV], nxt[GV];
  // the step's later kernels may launch now; they wait for this grid where needed
  asm volatile("griddepcontrol.launch_dependents;");
  int item = blockIdx.x, wave = 0, row = 0, nv = 0, l0 = 0;
  bool ok = false;
  const uint4* v = nullptr;
  if (item < nitems) {
    greedy_item<DT>(P, item, G, chunk, &row, &ok, &v, &nv, &l0);
    greedy_wave<DT>(v, nv, 0, cur);
  }
  // a batch without temperature-0 sequences: only the cluster kernel's work
  // flag is left to set (for sequences keyhist_kernel does not serve)
  // (checked only by CTAs whose first row is not on the greedy path)
  bool zt = ok;
  if (!__syncthreads_or(ok ? 1 : 0))
    for (int b = tid; b < P.B; b += NT) zt |= P.temp[b] == 0.0f;
  if (!__syncthreads_or(zt ? 1 : 0) && !P.greedy_only) {
    bool other = false;
    if (blockIdx.x == 0)
      for (int b = tid; b < P.B; b += NT) other |= !(P.fast_split && fast_seq(P, b));
    if (__syncthreads_or(other ? 1 : 0) && tid == 0) atomicOr(P.ws_work, 1u);
    return;
  }
  // the CTA's (item, wave) pairs form one stream: the next pair's loads are in
  // flight while the current one is reduced. Per thread: the running maximum,
  // the first vector holding it (and its contents), and a NaN flag.
  float mt = -INFINITY;
  int vb = -1;
  uint4 wb = make_uint4(0u, 0u, 0u, 0u);
  bool nanf = false;
  int nrow = row, nnv = nv, nl0 = l0;
  bool nok = ok;
  const uint4* nvp = v;
  while (item < nitems) {
    int nitem = item, nwave = wave + 1;
    if (nwave * WV >= nv) {
      nitem = item + (int)gridDim.x;
      nwave = 0;
      if (nitem < nitems) greedy_item<DT>(P, nitem, G, chunk, &nrow, &nok, &nvp, &nnv, &nl0);
    }
    if (nitem < nitems) greedy_wave<DT>(nitem == item ? v : nvp, nitem == item ? nv : nnv, nwave * WV, nxt);
    if (ok) {
#pragma unroll
      for (int q = 0; q < GV; ++q) {
        const int vi = wave * WV + tid + q * NT;
        const float vm = greedy_vmax<DT>(cur[q]);
        nanf |= vm != vm;
        if (vi < nv && vm > mt) {
          mt = vm;
          vb = vi;
          wb = cur[q];
        }
      }
    }
    if (nitem != item) {
      if (ok) {
        // the lowest index holding the maximum: within the first vector holding it
        uint32_t idx = UINT_MAX;
        if (vb >= 0 && mt < INFINITY) {
          const uint32_t ws[4] = {wb.x, wb.y, wb.z, wb.w};
          const uint32_t base = (uint32_t)(l0 + vb * PV);
#pragma unroll
          for (int h = 3; h >= 0; --h) {
            if constexpr (sizeof(DT) == 2) {
              if (__uint_as_float(ws[h] & 0xFFFF0000u) == mt) idx = base + 2 * h + 1;
              if (__uint_as_float(ws[h] << 16) == mt) idx = base + 2 * h;
            } else {
              if (__uint_as_float(ws[h]) == mt) idx = base + h;
            }
          }
        }
        const bool bad = nanf || mt == INFINITY;
        unsigned long long key = idx != UINT_MAX ? (((unsigned long long)okey(mt) << 32) | (uint32_t)~idx) : 0ull;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const unsigned long long o2 = __shfl_xor_sync(0xffffffffu, key, o);
          key = o2 > key ? o2 : key;
        }
        // one merge per warp and item, without a reply (the row's slot takes the
        // largest key); no block barrier, so every warp keeps its loads flowing
        const bool wbad = __any_sync(0xffffffffu, bad);
        if (lane_id() == 0) {
          if (wbad) atomicOr(&rflag[row], 1u);
          else if (key) atomicMax(&best[row], key);
        }
      } else if (!P.greedy_only && tid == 0 && item - row * G == 0 &&
                 !(P.fast_split && fast_seq(P, row / (P.K + 1))) &&
                 *reinterpret_cast<volatile unsigned int*>(P.ws_work) == 0u) {
        // rows of sampled sequences: the cluster kernel has work unless they all
        // go to keyhist_kernel (which raises the flag itself when it hands one back)
        atomicOr(P.ws_work, 1u);
      }
      mt = -INFINITY;
      vb = -1;
      nanf = false;
      row = nrow;
      ok = nok;
      v = nvp;
      nv = nnv;
      l0 = nl0;
    }
#pragma unroll
    for (int q = 0; q < GV; ++q) cur[q] = nxt[q];
    item = nitem;
    wave = nwave;
  }
  // the last CTA to finish writes the greedy sequences' outputs
  __shared__ int last_cta;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    last_cta = atomicAdd(done, 1u) == gridDim.x - 1u;
  }
  __syncthreads();
  if (last_cta) {
    __threadfence();
    for (int b = tid; b < P.B; b += NT) {
      if (greedy_seq(P, b)) {
        greedy_finalize_seq(P, b, best, rflag);
      } else if (P.greedy_only) {
        // no draft logits: a sequence off the greedy path is a data error
        for (int q = 0; q <= P.K; ++q) P.out_tokens[(size_t)b * (P.K + 1) + q] = -1;
        P.out_n[b] = -1;
      }
    }
    if (tid == 0) *done = 0u;
  }
}


// Decode-loop handoff after a verify step: each sequence's last emitted token
// becomes its next input token, its length grows by the tokens emitted (n + 1;
// nothing on a data error), and the Philox offset in device memory advances by
// one for the next step. Runs after every kernel of the step (stream order).
__global__ void handoff_kernel(const int32_t* out_tokens, const int32_t* out_n, int B, int K,
                               int32_t* next_token, int32_t* seq_len, uint64_t* offset) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) {
    const int n = out_n[b];
    if (next_token) next_token[b] = n >= 0 ? out_tokens[(size_t)b * (K + 1) + n] : -1;
    if (seq_len && n >= 0) seq_len[b] += n + 1;
  }
  if (b == 0) *offset += 1ull;
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
struct Geometry {
  int C, slice, ept, slot_elems, NS;
  size_t smem;
};

// Cluster size: the smallest C (1..16) whose row slice fits a ~20 KB slot, else
// 16. Four slots (two paired units) when two CTAs fit an SM, else as many as
// fit one CTA per SM.
static Geometry geometry(int V, int es) {
  Geometry g{};
  const size_t fixed = SHARED_BYTES + H_BYTES + G_BYTES;
  for (int C = 1; C <= 16; ++C) {
    int slice = (V + C - 1) / C;
    slice = (slice + 7) & ~7;
    if ((long long)(C - 1) * slice >= V) continue;
    int per = (slice + NT - 1) / NT;
    int words = (per * es + 3) / 4;
    words |= 1;                                   // odd word stride: no bank conflicts
    const int ept = words * 4 / es;
    const size_t slot = (size_t)NT * ept * es;
    g.C = C;
    g.slice = slice;
    g.ept = ept;
    g.slot_elems = NT * ept;
    if (slot <= 20 * 1024 || C == 16) break;
  }
  const size_t slot = (size_t)g.slot_elems * es;
  g.NS = NSMAX;
  while (g.NS > 2 && fixed + g.NS * slot > 227 * 1024) --g.NS;
  g.smem = fixed + (size_t)g.NS * slot;
  if (g.smem > 227 * 1024 || g.ept > 255) g.smem = 0;
  return g;
}

static LaunchCache g_launch_cache;

// Raises (never lowers) a kernel's dynamic shared-memory limit on the current
// device: launches with different sizes share the attribute.
static cudaError_t ensure_smem_limit(const void* fn, size_t smem) {
  cudaFuncAttributes fa;
  cudaError_t r = cudaFuncGetAttributes(&fa, fn);
  if (r != cudaSuccess) return r;
  if ((size_t)fa.maxDynamicSharedSizeBytes >= smem) return cudaSuccess;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

// Resident grid of a persistent kernel on the current device (SMs times the CTAs
// of `threads` threads and `smem` dynamic shared memory that fit one SM), with the
// kernel's dynamic shared-memory limit raised on this device first.
static cudaError_t resident_grid(const void* fn, int threads, size_t smem, int* grid) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return g_launch_cache.get(dev, fn, smem, threads, grid, [&](int* v) {
    cudaError_t r;
    if ((r = ensure_smem_limit(fn, smem)) != cudaSuccess) return r;
    int sms = 0, per = 0;
    if ((r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return r;
    if ((r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, fn, threads, smem)) != cudaSuccess) return r;
    *v = (sms > 1 ? sms : 1) * (per > 1 ? per : 1);
    return cudaSuccess;
  });
}
static cudaError_t keyhist_grid(void (*fn)(const Params, int), int* grid) {
  return resident_grid(reinterpret_cast<const void*>(fn), KT, KH_SMEM, grid);
}

template <typename DT, int MODE>
static cudaError_t launch(const Params& p, const Geometry& g, cudaStream_t st) {
  auto kern = sv_kernel<DT, MODE>;
  cudaError_t e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)g.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // verify calls: may start while the step's earlier kernels finish (it waits for
  // them with griddepcontrol.wait before reading their results)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (MODE == MODE_VERIFY && p.greedy_split) ? 2 : 1;
  // clusters that fit the device at once, with the kernel's attributes set on this
  // device (cached per device, cluster size and shared memory)
  int max_clusters = 0;
  e = g_launch_cache.get(dev, reinterpret_cast<const void*>(kern), g.smem, g.C, &max_clusters,
                         [&](int* v) {
                           cudaError_t r = ensure_smem_limit(reinterpret_cast<const void*>(kern), g.smem);
                           if (r != cudaSuccess) return r;
                           r = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                           if (r != cudaSuccess) return r;
                           cudaLaunchConfig_t q = cfg;
                           q.gridDim = dim3((unsigned)g.C, 1, 1);
                           int n = 0;
                           r = cudaOccupancyMaxActiveClusters(&n, kern, &q);
                           *v = n > 0 ? n : 1;
                           return r;
                         });
  if (e != cudaSuccess) return e;
  const int ncl = min(max_clusters, p.nunits);
  cfg.gridDim = dim3((unsigned)(ncl * g.C), 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, p);
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
  p.C = g->C;
  p.slice = g->slice;
  p.ept = g->ept;
  p.slot_elems = g->slot_elems;
  p.NS = g->NS;
  return g->smem != 0;
}

static sv_status do_launch(int mode, sv_dtype dt, const Params& p, const Geometry& g, cudaStream_t st) {
  cudaError_t e;
  if (dt == SV_BF16) {
    if (mode == MODE_VERIFY) e = launch<__nv_bfloat16, MODE_VERIFY>(p, g, st);
    else if (mode == MODE_PROBS) e = launch<__nv_bfloat16, MODE_PROBS>(p, g, st);
    else e = launch<__nv_bfloat16, MODE_SAMPLE>(p, g, st);
  } else {
    if (mode == MODE_VERIFY) e = launch<float, MODE_VERIFY>(p, g, st);
    else if (mode == MODE_PROBS) e = launch<float, MODE_PROBS>(p, g, st);
    else e = launch<float, MODE_SAMPLE>(p, g, st);
  }
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

static bool aligned(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

extern "C" {

// Workspace layout: [units u64 x B(K+1)][tickets u32 x B, padded to 16][error u32,
// padded to 16][greedy best u64 x B(K+1)][greedy chunk counters u32 x B(K+1)]
// [greedy flags u32 x B(K+1)], padded to 16; then for the per-row kernels
// [hand-back flags u32 x B, padded][row results x B(2K+1)][work counter, CTAs
// done: 16 bytes][kept-token lists u32 x B(K+1) x 256][sequence order i32 x B,
// padded]; all of it zero between calls.
size_t spec_verify_workspace_bytes(int B, int K) {
  if (B < 1 || K < 1) return 0;
  const size_t rows = (size_t)B * (K + 1);
  const size_t tickets = ((size_t)B * sizeof(unsigned int) + 15) & ~(size_t)15;
  const size_t head = rows * 8 + tickets + 16 + rows * 8 + rows * 4 + rows * 4;
  // keyhist_kernel: hand-back flags, row results, work counter, kept-token lists
  return ((head + 15) & ~(size_t)15) + tickets + (size_t)B * (2 * K + 1) * sizeof(KhRow) + 16 +
         rows * KH_KCAP * sizeof(uint32_t) + tickets;
}

static sv_status verify_impl(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                             const int32_t* draft_tokens, const float* temperature,
                             const int32_t* top_k, const float* top_p, uint64_t philox_seed,
                             uint64_t philox_offset, const uint64_t* offset_ptr, int B, int K,
                             int V, int32_t* out_tokens, int32_t* out_n_accepted, void* workspace,
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
  p.offset_ptr = offset_ptr;
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
  const size_t rows = (size_t)p.nunits;
  char* w2 = ws + rows * 8 + (((size_t)B * 4 + 15) & ~(size_t)15);
  p.ws_error = reinterpret_cast<unsigned int*>(w2);
  p.ws_work = reinterpret_cast<unsigned int*>(w2 + 4);
  p.ws_done = reinterpret_cast<unsigned int*>(w2 + 8);
  p.ws_best = reinterpret_cast<unsigned long long*>(w2 + 16);
  p.ws_rcnt = reinterpret_cast<unsigned int*>(w2 + 16 + rows * 8);
  p.ws_rflag = reinterpret_cast<unsigned int*>(w2 + 16 + rows * 12);
  {
    const size_t tickets = ((size_t)B * sizeof(unsigned int) + 15) & ~(size_t)15;
    const size_t head = rows * 8 + tickets + 16 + rows * 8 + rows * 4 + rows * 4;
    char* w3 = ws + ((head + 15) & ~(size_t)15);
    p.ws_fb = reinterpret_cast<unsigned int*>(w3);
    p.ws_rowres = reinterpret_cast<KhRow*>(w3 + tickets);
    char* w4 = w3 + tickets + (size_t)B * (2 * K + 1) * sizeof(KhRow);
    p.ws_fnext = reinterpret_cast<unsigned int*>(w4);
    p.ws_fdone = reinterpret_cast<unsigned int*>(w4 + 4);
    p.ws_lists = reinterpret_cast<uint32_t*>(w4 + 16);
    p.ws_perm = reinterpret_cast<int*>(w4 + 16 + rows * KH_KCAP * sizeof(uint32_t));
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // temperature-0 units: streaming reduction; the cluster kernel takes the rest
  // (unaligned rows: the cluster kernel serves every unit)
  if (p.bulk_ok) {
    // without draft logits every sequence must be greedy (others are data
    // errors), so the greedy kernel alone serves the batch
    p.greedy_only = draft_logits == nullptr ? 1 : 0;
    // sampled bf16 sequences: one-pass key-histogram kernel, one CTA per row;
    // batches of fewer units than the cluster kernel runs clusters keep each
    // row spread over a cluster of SMs instead
    p.fast_split = (draft_logits != nullptr && (long long)B * (K + 1) >= 16) ? 1 : 0;
    const int PV = 16 / (int)es;
    const int cmax = GW * GV * NT * PV;
    const int G = (V + cmax - 1) / cmax;
    int chunk = (V + G - 1) / G;
    chunk = (chunk + PV - 1) / PV * PV;
    const long long nitems = (long long)rows * G;
    int gblocks = 0;
    if (resident_grid(reinterpret_cast<const void*>(greedy_kernel<__nv_bfloat16>), NT, 0, &gblocks) !=
        cudaSuccess)
      return SV_ERR_CUDA;
    const unsigned grid = (unsigned)(nitems < (long long)gblocks ? nitems : (long long)gblocks);
    // fp32 rows: the sampled sequences' processing order for fstream_kernel, set
    // before the step's other kernels start (they launch after this one ends)
    if (dtype == SV_F32 && p.fast_split && !p.greedy_only) {
      fs_order_kernel<<<1, 1024, 0, st>>>(p);
      if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    }
    if (dtype == SV_BF16)
      greedy_kernel<__nv_bfloat16><<<grid, NT, 0, st>>>(p, G, chunk, (int)nitems, p.ws_best, p.ws_rflag, p.ws_rcnt);
    else
      greedy_kernel<float><<<grid, NT, 0, st>>>(p, G, chunk, (int)nitems, p.ws_best, p.ws_rflag, p.ws_rcnt);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    p.greedy_split = 1;
    if (p.greedy_only) return SV_OK;
    if (p.fast_split) {
      // sampled sequences, one CTA per row: the key-histogram kernel for bf16 rows,
      // the fp32 streaming kernel for fp32 rows
      const bool bf = dtype == SV_BF16;
      void (*fk)(const Params, int) = bf ? keyhist_kernel : fstream_kernel;
      const size_t fsm = bf ? KH_SMEM : FS_SMEM;
      int kblocks = 0;
      if (resident_grid(reinterpret_cast<const void*>(fk), KT, fsm, &kblocks) != cudaSuccess)
        return SV_ERR_CUDA;
      const int kitems = B * (2 * K + 1);
      const int kgrid = kitems < kblocks ? kitems : kblocks;
      // starts while greedy_kernel runs (it reads nothing greedy_kernel writes, and
      // waits for it before finishing, so the cluster kernel sees both)
      cudaLaunchConfig_t kc = {};
      kc.gridDim = dim3((unsigned)kgrid, 1, 1);
      kc.blockDim = dim3(KT, 1, 1);
      kc.dynamicSmemBytes = fsm;
      kc.stream = st;
      cudaLaunchAttribute ka[1];
      ka[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      ka[0].val.programmaticStreamSerializationAllowed = 1;
      kc.attrs = ka;
      kc.numAttrs = 1;
      if (cudaLaunchKernelEx(&kc, fk, p, kitems) != cudaSuccess) return SV_ERR_CUDA;
    }
  }
  return do_launch(MODE_VERIFY, dtype, p, g, st);
}

sv_status spec_verify(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      const int32_t* draft_tokens, const float* temperature, const int32_t* top_k,
                      const float* top_p, uint64_t philox_seed, uint64_t philox_offset, int B,
                      int K, int V, int32_t* out_tokens, int32_t* out_n_accepted, void* workspace,
                      size_t workspace_bytes, void* stream) {
  return verify_impl(target_logits, draft_logits, dtype, draft_tokens, temperature, top_k, top_p,
                     philox_seed, philox_offset, nullptr, B, K, V, out_tokens, out_n_accepted,
                     workspace, workspace_bytes, stream);
}

sv_status spec_verify_step(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                           const int32_t* draft_tokens, const float* temperature,
                           const int32_t* top_k, const float* top_p, uint64_t philox_seed,
                           uint64_t* philox_offset, int B, int K, int V, int32_t* out_tokens,
                           int32_t* out_n_accepted, int32_t* next_token, int32_t* seq_len,
                           void* workspace, size_t workspace_bytes, void* stream) {
  if (!philox_offset) return SV_ERR_NULL;
  if (!aligned(philox_offset, 8) || (next_token && !aligned(next_token, 4)) ||
      (seq_len && !aligned(seq_len, 4)))
    return SV_ERR_ALIGN;
  const sv_status s = verify_impl(target_logits, draft_logits, dtype, draft_tokens, temperature,
                                  top_k, top_p, philox_seed, 0, philox_offset, B, K, V, out_tokens,
                                  out_n_accepted, workspace, workspace_bytes, stream);
  if (s != SV_OK) return s;
  handoff_kernel<<<(B + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      out_tokens, out_n_accepted, B, K, next_token, seq_len, philox_offset);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // bf16 rows, 16-byte aligned, at least 16 rows: the per-row code of the sampled
  // verify path serves every row it can; the cluster kernel takes the rows it marks
  p.fast_split = (dtype == SV_BF16 && p.bulk_ok && R >= 16) ? 1 : 0;
  if (p.fast_split) {
    int grid = 0;
    if (keyhist_grid(keyhist_probs_kernel, &grid) != cudaSuccess) return SV_ERR_CUDA;
    keyhist_probs_kernel<<<R < grid ? R : grid, KT, KH_SMEM, st>>>(p, R);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  }
  return do_launch(MODE_PROBS, dtype, p, g, st);
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // bf16 rows, 16-byte aligned, at least 16 rows: the key-histogram sampler serves
  // every row it can; the cluster kernel takes the rows it marks
  p.fast_split = (dtype == SV_BF16 && p.bulk_ok && (long long)B * K >= 16) ? 1 : 0;
  if (p.fast_split) {
    int sblocks = 0;
    if (keyhist_grid(keyhist_sample_kernel, &sblocks) != cudaSuccess) return SV_ERR_CUDA;
    const int items = B * K;
    keyhist_sample_kernel<<<items < sblocks ? items : sblocks, KT, KH_SMEM, st>>>(p, items);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  }
  return do_launch(MODE_SAMPLE, dtype, p, g, st);
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

// Test hook for the per-device launch cache, no GPU needed: eight host threads
// look up two kernels on two fake devices whose queries report different SM
// counts (152 and 132, two CTAs per SM). out[0..3] = grids of (device 0, kernel
// A), (device 1, A), (device 0, B), (device 1, B); out[4] = cache entries (4);
// out[5] = 1 if every thread saw the same values. Returns 0.
int sv_test_launch_cache(int* out) {
  LaunchCache cache;
  static const char fa = 0, fb = 0;
  const void* fns[2] = {&fa, &fb};
  int seen[8][4];
  std::vector<std::thread> th;
  for (int t = 0; t < 8; ++t)
    th.emplace_back([&, t]() {
      for (int r = 0; r < 4; ++r) {
        const int j = (r + t) & 3, dev = j & 1, f = j >> 1;
        int v = 0;
        cache.get(dev, fns[f], 1024, 512, &v, [&](int* q) {
          *q = (dev == 0 ? 152 : 132) * 2 + f;
          return cudaSuccess;
        });
        seen[t][j] = v;
      }
    });
  for (auto& x : th) x.join();
  for (int j = 0; j < 4; ++j) out[j] = seen[0][j];
  out[4] = (int)cache.size();
  int same = 1;
  for (int t = 1; t < 8; ++t)
    for (int j = 0; j < 4; ++j) same &= seen[t][j] == seen[0][j];
  out[5] = same;
  return 0;
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

int sv_version(void) { return 300; }

#ifdef SV_TRACE
int sv_trace_reset(void) {
  static unsigned long long zero[64 * 32 + 16];
  return cudaMemcpyToSymbol(g_trace, zero, sizeof(zero)) == cudaSuccess ? 0 : 1;
}
int kh_trace_reset(void) {
  static unsigned long long zero[8192 * 8];
  if (cudaMemcpyToSymbol(g_khtrace, zero, sizeof(zero)) != cudaSuccess) return 1;
  if (cudaMemcpyToSymbol(g_khheavy, zero, sizeof(unsigned long long)) != cudaSuccess) return 1;
  return cudaMemcpyToSymbol(g_kftrace, zero, 1024 * 8 * sizeof(unsigned long long)) == cudaSuccess ? 0 : 1;
}
unsigned long long kh_heavy_count(void) {
  unsigned long long v = 0;
  cudaMemcpyFromSymbol(&v, g_khheavy, sizeof(v));
  return v;
}
int kf_trace_copy(unsigned long long* host, size_t n) {
  if (n > 1024 * 8) n = 1024 * 8;
  return cudaMemcpyFromSymbol(host, g_kftrace, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : 1;
}
int kh_trace_copy(unsigned long long* host, size_t n) {
  if (n > 8192 * 8) n = 8192 * 8;
  return cudaMemcpyFromSymbol(host, g_khtrace, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : 1;
}
int sv_trace_copy(unsigned long long* host, size_t n) {
  if (n > 64 * 32 + 16) n = 64 * 32 + 16;
  return cudaMemcpyFromSymbol(host, g_trace, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : 1;
}
#endif

}  // extern "C"
