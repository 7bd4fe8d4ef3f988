// LM-head logits on the 5th-generation tensor cores, and the verify step fed from
// hidden states (C ABI in include/spec_lm_head.h).
//
// Z[M][N] = H[M][d] . W[N][d]^T with bf16 operands and an fp32 accumulator: the
// output projection that ends a decode step ("Apple Silikon İçin Cihaz Üstü
// Çıkarımı Optimize Etme", perplexity.coolkeypoint.com, decode section).
//
// A persistent grid (one CTA per SM) walks the 128 x 256 output tiles, the
// column-tile index outer, so the CTAs at work at any time share few W tiles and
// W is read from HBM about once. Warp roles: warp 0 issues the TMA loads of both
// K-major operands (128-byte swizzle, one 64-element K slice per stage) into a
// 4-stage ring, running ahead across tiles; warp 1 allocates two 256-column fp32
// TMEM accumulators and one of its threads issues tcgen05.mma (M = 128, N = 256,
// K = 16) into them in turn; warps 2-5 read a finished accumulator back with
// tcgen05.ld (each warp its quarter of the TMEM lanes, i.e. 32 output rows) while
// the next tile is being multiplied into the other one, and either store fp32
// rows or, for the greedy verify step, reduce them to each row's maximum and the
// lowest column holding it, so that the logits never reach memory. Every wait is
// bounded: a timeout sets the caller's flag, the CTA lets its issued copies and
// MMAs land and frees its TMEM before it returns.
//
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spec_lm_head.h"
#include "launch_cache.h"

namespace svlm {

constexpr int BM = 128, BN = 256, BK = 64;   // BK bf16 = 128 bytes: one swizzle row
constexpr int NS = 4;                          // pipeline stages
constexpr int STAGE_A = BM * BK * 2, STAGE_B = BN * BK * 2;   // 16 KB and 32 KB
constexpr int TMEM_COLS = 2 * BN;              // two fp32 accumulators, 128 lanes x 256 columns each
constexpr int NEPI = 4;                        // epilogue warps (one TMEM lane quarter each)
constexpr int NTHREADS = 64 + 32 * NEPI;       // TMA warp, MMA warp, epilogue warps
constexpr uint64_t WAIT_NS = 200ull * 1000 * 1000;

struct __align__(8) Ctl {
  unsigned long long full[NS], empty[NS];      // stage loaded / stage consumed by the MMAs
  unsigned long long acc_full[2], acc_empty[2];   // accumulator finished / read back
  unsigned long long done;                     // every MMA of the CTA finished
  uint32_t taddr;
  int err;
};
constexpr int CTL_BYTES = ((int)sizeof(Ctl) + 15) & ~15;
constexpr int STG_BYTES = NEPI * 32 * 33 * 4;   // EPI_STORE: one 32 x 32 transpose block per epilogue warp
constexpr int SMEM_BYTES = 1024 /* alignment slack */ + NS * (STAGE_A + STAGE_B) + CTL_BYTES + STG_BYTES;

__device__ __forceinline__ uint32_t sa(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bar_init(unsigned long long* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_expect(unsigned long long* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool bar_try(unsigned long long* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(sa(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bar_arrive(unsigned long long* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(b)) : "memory");
}
// Waits for phase `parity` of b for at most WAIT_NS; false on timeout.
__device__ __forceinline__ bool bar_wait(unsigned long long* b, uint32_t parity) {
  if (bar_try(b, parity)) return true;
  const uint64_t t0 = now_ns();
  while (!bar_try(b, parity))
    if (now_ns() - t0 > WAIT_NS) return false;
  return true;
}
// 2-D tiled TMA load of the box at (x = K coordinate, y = row); x is a multiple
// of 64 elements, so x * 2 bytes is 16-byte aligned.
__device__ __forceinline__ void tma_load(void* dst, const CUtensorMap* map, int x, int y,
                                         unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(sa(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(sa(bar))
      : "memory");
}
// Shared-memory matrix descriptor of a K-major operand with 128-byte swizzle:
// start address, leading byte offset (unused with this swizzle), stride byte
// offset 1024 (eight 128-byte rows), descriptor version 1, swizzle code 2. Stage
// bases are 1024-byte aligned, so the base offset field stays 0.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Instruction descriptor (kind::f16): fp32 D (bits 4-5 = 1), bf16 A and B (bits
// 7-9 and 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma(uint32_t taddr, uint64_t a, uint64_t b, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(taddr),
      "l"(a), "l"(b), "r"(IDESC), "r"(accum)
      : "memory");
}
// Arrives on bar once every tcgen05 operation this thread issued before is done.
__device__ __forceinline__ void commit(unsigned long long* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sa(bar))
               : "memory");
}

// Epilogues: EPI_STORE writes the fp32 logit tile to Z; EPI_ARGMAX reduces each
// row of the tile to (order key of its maximum << 32 | ~lowest column holding
// it) and merges that into keys[row] with a 64-bit atomicMax, so the largest key
// over all column tiles names the row's first maximum. NaN takes the largest
// order key, so a row holding one reads as NaN.
constexpr int EPI_STORE = 0, EPI_ARGMAX = 1;

// Order-preserving 32-bit key of an fp32 value (NaN: 0xFFFFFFFF).
__device__ __forceinline__ uint32_t order_key(uint32_t u) {
  if (__uint_as_float(u) != __uint_as_float(u)) return 0xFFFFFFFFu;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
constexpr uint32_t KEY_NEG_INF = 0x007FFFFFu;   // order_key(-inf)
constexpr uint32_t KEY_POS_INF = 0xFF800000u;   // order_key(+inf)

template <int EPI>
__global__ void __launch_bounds__(NTHREADS, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap mapH, const __grid_constant__ CUtensorMap mapW,
                   float* __restrict__ Z, unsigned long long* __restrict__ keys, int M, int N, int d,
                   int32_t* flag) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* sA = smem;
  unsigned char* sB = smem + NS * STAGE_A;
  Ctl& C = *reinterpret_cast<Ctl*>(smem + NS * (STAGE_A + STAGE_B));
  float* stg = reinterpret_cast<float*>(smem + NS * (STAGE_A + STAGE_B) + CTL_BYTES);
  volatile int* err = &C.err;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = (M + BM - 1) / BM;
  const long long ntiles = (long long)mt * ((N + BN - 1) / BN);
  const int nk = d / BK;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      bar_init(&C.full[s], 1);
      bar_init(&C.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      bar_init(&C.acc_full[b], 1);
      bar_init(&C.acc_empty[b], 32 * NEPI);
    }
    bar_init(&C.done, 1);
    C.err = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {   // the whole warp allocates (and later frees) the accumulators
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sa(&C.taddr)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  }
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t taddr = C.taddr;

  // K slices loaded and consumed are counted over all tiles of the CTA: slice
  // number `it` uses stage it % NS in its (it / NS)-th round
  long long issued = 0;
  if (warp == 0) {
    if (lane == 0) {
      long long it = 0;
      for (long long t = blockIdx.x; t < ntiles && !*err; t += gridDim.x) {
        const int m0 = (int)(t % mt) * BM, n0 = (int)(t / mt) * BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = (int)(it % NS);
          // reuse of stage s waits for the MMAs of its previous slice
          if (it >= NS && !bar_wait(&C.empty[s], (uint32_t)((it / NS - 1) & 1))) {
            atomicExch(&C.err, 1);
            break;
          }
          if (*err) break;
          bar_expect(&C.full[s], STAGE_A + STAGE_B);
          tma_load(sA + s * STAGE_A, &mapH, kb * BK, m0, &C.full[s]);
          tma_load(sB + s * STAGE_B, &mapW, kb * BK, n0, &C.full[s]);
          issued = it + 1;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      long long it = 0;
      int j = 0;   // tiles of this CTA so far; tile j accumulates into buffer j & 1
      for (long long t = blockIdx.x; t < ntiles && !*err; t += gridDim.x, ++j) {
        const int buf = j & 1;
        // the epilogue has read this buffer's previous tile
        if (j >= 2 && !bar_wait(&C.acc_empty[buf], (uint32_t)((j / 2 - 1) & 1))) {
          atomicExch(&C.err, 1);
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t tacc = taddr + (uint32_t)(buf * BN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = (int)(it % NS);
          if (!bar_wait(&C.full[s], (uint32_t)((it / NS) & 1))) {
            atomicExch(&C.err, 1);
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t a0 = sa(sA + s * STAGE_A), b0 = sa(sB + s * STAGE_B);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)   // 16 bf16 = 32 bytes along K per instruction
            mma(tacc, sdesc(a0 + k * 32), sdesc(b0 + k * 32), (kb | k) != 0);
          commit(&C.empty[s]);
        }
        if (!ok) break;
        commit(&C.acc_full[buf]);
      }
      commit(&C.done);
    }
  } else {
    // epilogue: warp w may read TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31
    const int q = warp & 3;
    int j = 0;
    for (long long t = blockIdx.x; t < ntiles; t += gridDim.x, ++j) {
      const int buf = j & 1;
      const bool got = bar_wait(&C.acc_full[buf], (uint32_t)((j / 2) & 1)) && !*err;
      // tcgen05.ld is warp-collective: the whole warp takes the same branch
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) atomicExch(&C.err, 1);
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int m0 = (int)(t % mt) * BM, n0 = (int)(t / mt) * BN;
      const int row = m0 + q * 32 + lane;
      uint32_t bkey = 0u, bcol = 0u;   // EPI_ARGMAX: the thread's best order key and its column
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        const uint32_t ta = taddr + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + c * 32);
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
            "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
            "[%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
              "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
              "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
              "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
            : "r"(ta));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const int col = n0 + c * 32;
        if (EPI == EPI_ARGMAX) {
          // ascending columns and a strict comparison: the first maximum is kept
          const int lim = min(32, N - col);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const uint32_t key = order_key(r[jj]);
            if (jj < lim && key > bkey) {
              bkey = key;
              bcol = (uint32_t)(col + jj);
            }
          }
        } else if (col < N) {
          // a lane holds one row's 32 columns; through the warp's block of shared
          // memory (row stride 33: no bank conflicts either way) each store
          // instruction writes 32 consecutive columns of one row instead
          float* st = stg + q * (32 * 33);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) st[lane * 33 + jj] = __uint_as_float(r[jj]);
          __syncwarp();
          const int cl = col + lane;
          const int rb = m0 + q * 32, nr = min(32, M - rb);
          for (int i = 0; i < nr; ++i)
            if (cl < N) Z[(size_t)(rb + i) * N + cl] = st[i * 33 + lane];
          __syncwarp();
        }
      }
      // the buffer may take the next tile once every epilogue thread has read it
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      bar_arrive(&C.acc_empty[buf]);
      if (EPI == EPI_ARGMAX && row < M && bkey != 0u)
        atomicMax(keys + row, ((unsigned long long)bkey << 32) | (unsigned long long)(~bcol));
    }
  }
  __syncwarp();
  __syncthreads();
  // before TMEM is freed: every MMA issued has finished (the MMA thread's last
  // commit) and, after a timeout, the copies issued but never consumed have landed
  if (tid == 0) bar_wait(&C.done, 0u);
  if (warp == 0 && lane == 0 && *err) {
    for (long long it = issued > NS ? issued - NS : 0; it < issued; ++it)
      bar_wait(&C.full[it % NS], (uint32_t)((it / NS) & 1));
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(TMEM_COLS)
                 : "memory");
  }
  if (tid == 0 && *err) atomicExch(flag, 1);
}

// Greedy acceptance of sequence b from its K+1 row keys (one thread per
// sequence): the drafted tokens are kept while each equals its row's first
// maximum; the first row that disagrees (or row K after K matches) gives the last
// token. A row whose maximum is NaN or +inf or whose logits are all -inf, or a
// drafted token outside [0, V), makes the sequence a data error (n = -1, every
// token -1). The keys are zeroed for the next call.
__global__ void lm_greedy_kernel(unsigned long long* __restrict__ keys, const int32_t* __restrict__ dtok,
                                 int B, int K, int V, int32_t* __restrict__ out_tokens,
                                 int32_t* __restrict__ out_n) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int K1 = K + 1;
  unsigned long long* kb = keys + (size_t)b * K1;
  const int32_t* db = dtok + (size_t)b * K;
  bool bad = false;
  for (int q = 0; q < K; ++q) bad |= db[q] < 0 || db[q] >= V;
  int n = 0;
  int last = -1;
  for (int i = 0; i < K1; ++i) {
    const unsigned long long key = kb[i];
    kb[i] = 0ull;
    const uint32_t ok = (uint32_t)(key >> 32);
    bad |= ok <= KEY_NEG_INF || ok >= KEY_POS_INF;
    const int amax = (int)~(uint32_t)key;
    if (n == i && last < 0) {
      if (i < K && db[i] == amax) ++n;
      else last = amax;
    }
  }
  int32_t* ob = out_tokens + (size_t)b * K1;
  for (int q = 0; q < K1; ++q) ob[q] = bad ? -1 : (q < n ? db[q] : (q == n ? last : -1));
  out_n[b] = bad ? -1 : n;
}

typedef CUresult (*EncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiled>(p);
  }
  return fn;
}

// rows x d bf16, row-major; boxes of 64 x box_rows with 128-byte swizzle; rows
// past the end read as zero
static bool make_map(CUtensorMap* map, const void* base, int rows, int d, int box_rows) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static sv::LaunchCache g_lm_cache;

// Encodes the operand maps and launches one GEMM (arguments already checked).
template <int EPI>
static sv_status launch_gemm(const void* hidden, const void* weight, int M, int N, int d, float* logits,
                             unsigned long long* keys, int32_t* flag, cudaStream_t stream) {
  CUtensorMap mh, mw;
  if (!make_map(&mh, hidden, M, d, BM) || !make_map(&mw, weight, N, d, BN)) return SV_ERR_CUDA;
  // the kernel's shared-memory limit, raised once per device
  int dev = 0, done = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      g_lm_cache.get(dev, reinterpret_cast<const void*>(lm_head_kernel<EPI>), SMEM_BYTES, 0, &done, [](int* v) {
        *v = 1;
        return cudaFuncSetAttribute(lm_head_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    SMEM_BYTES);
      }) != cudaSuccess)
    return SV_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return SV_ERR_CUDA;
  const long long tiles = (long long)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
  lm_head_kernel<EPI><<<grid, NTHREADS, SMEM_BYTES, stream>>>(mh, mw, logits, keys, M, N, d, flag);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace svlm

sv_status spec_lm_head_logits(const void* hidden, const void* weight, int M, int N, int d, float* logits,
                              int32_t* flag, void* stream) {
  using namespace svlm;
  if (!hidden || !weight || !logits || !flag) return SV_ERR_NULL;
  if (M < 1 || M > 2147483647 - BM || N < 1 || N > 65535 * BN || d < BK || d > 65536 || d % BK)
    return SV_ERR_SHAPE;
  if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(logits, 4) || !aligned(flag, 4))
    return SV_ERR_ALIGN;
  return svlm::launch_gemm<svlm::EPI_STORE>(hidden, weight, M, N, d, logits, nullptr, flag,
                                            static_cast<cudaStream_t>(stream));
}

sv_status spec_verify_from_hidden(const void* hidden_target, const void* weight_target, int d,
                                  const void* hidden_draft, const void* weight_draft, int d_draft,
                                  const int32_t* draft_tokens, const float* temperature, const int32_t* top_k,
                                  const float* top_p, uint64_t philox_seed, uint64_t philox_offset, int B, int K,
                                  int V, float* logits_scratch, int32_t* flag, int32_t* out_tokens,
                                  int32_t* out_n_accepted, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  // every argument is checked here, so that an error launches nothing
  if (!hidden_target || !weight_target || !logits_scratch || !flag || !draft_tokens || !temperature ||
      !top_k || !top_p || !out_tokens || !out_n_accepted || !workspace)
    return SV_ERR_NULL;
  if ((hidden_draft == nullptr) != (weight_draft == nullptr)) return SV_ERR_NULL;
  const auto bad_d = [](int dd) { return dd < svlm::BK || dd > 65536 || dd % svlm::BK != 0; };
  if (B < 1 || B > 65535 || K < 1 || K > 16 || V < 2 || V > 262144 || bad_d(d) ||
      (hidden_draft && bad_d(d_draft)))
    return SV_ERR_SHAPE;
  if (!svlm::aligned(logits_scratch, 16) || !svlm::aligned(hidden_target, 16) ||
      !svlm::aligned(weight_target, 16) || !svlm::aligned(flag, 4) ||
      (hidden_draft && (!svlm::aligned(hidden_draft, 16) || !svlm::aligned(weight_draft, 16))))
    return SV_ERR_ALIGN;
  if (workspace_bytes < spec_verify_workspace_bytes(B, K)) return SV_ERR_WORKSPACE;
  float* zt = logits_scratch;
  float* zd = logits_scratch + (size_t)B * (K + 1) * V;
  sv_status s = spec_lm_head_logits(hidden_target, weight_target, B * (K + 1), V, d, zt, flag, stream);
  if (s != SV_OK) return s;
  if (hidden_draft) {
    s = spec_lm_head_logits(hidden_draft, weight_draft, B * K, V, d_draft, zd, flag, stream);
    if (s != SV_OK) return s;
  }
  return spec_verify(zt, hidden_draft ? zd : nullptr, SV_F32, draft_tokens, temperature, top_k, top_p,
                     philox_seed, philox_offset, B, K, V, out_tokens, out_n_accepted, workspace,
                     workspace_bytes, stream);
}

sv_status spec_verify_greedy_from_hidden(const void* hidden_target, const void* weight, int d,
                                         const int32_t* draft_tokens, int B, int K, int V, int32_t* flag,
                                         int32_t* out_tokens, int32_t* out_n_accepted, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  if (!hidden_target || !weight || !draft_tokens || !flag || !out_tokens || !out_n_accepted || !workspace)
    return SV_ERR_NULL;
  if (B < 1 || B > 65535 || K < 1 || K > 16 || V < 2 || V > 262144 || d < svlm::BK || d > 65536 ||
      d % svlm::BK != 0)
    return SV_ERR_SHAPE;
  if (!svlm::aligned(hidden_target, 16) || !svlm::aligned(weight, 16) || !svlm::aligned(draft_tokens, 4) ||
      !svlm::aligned(flag, 4) || !svlm::aligned(out_tokens, 4) || !svlm::aligned(out_n_accepted, 4))
    return SV_ERR_ALIGN;
  if (!svlm::aligned(workspace, 16) || workspace_bytes < spec_verify_workspace_bytes(B, K))
    return SV_ERR_WORKSPACE;
  // the row keys use the workspace's first B(K+1) 64-bit words (zero between calls)
  unsigned long long* keys = static_cast<unsigned long long*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const sv_status s = svlm::launch_gemm<svlm::EPI_ARGMAX>(hidden_target, weight, B * (K + 1), V, d, nullptr,
                                                         keys, flag, st);
  if (s != SV_OK) return s;
  svlm::lm_greedy_kernel<<<(B + 127) / 128, 128, 0, st>>>(keys, draft_tokens, B, K, V, out_tokens,
                                                         out_n_accepted);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
