// Chunked Gated Delta Rule prefill for sm_103a.
//
// One CTA (128 threads, 4 warps) owns one (sequence, sab head) unit and walks
// its 64-token chunks in order.  For a chunk with rows i, j = 0..63, raw bf16
// tiles K, Q (q/k head) and V (v head), gates g, beta and the state S entering
// the chunk (Dv x Dk fp32, row = value index), the chunk-parallel form of the
// delta rule (Yang et al., "Parallelizing Linear Transformers with the Delta Rule
// over Sequence Length"; gated as in "Gated Delta Networks") is evaluated as:
//
//   G = cumsum(log g),  gam_i = e^{G_i},  d_j = e^{G_last - G_j}
//   rk_i, rq_i = 1/sqrt(|k_i|^2 + 1e-6), 1/sqrt(|q_i|^2 + 1e-6)  (1 without L2 norm)
//   A_ij = beta_i e^{G_i - G_j} rk_i rk_j (k_i . k_j)          (j < i)
//   T    = (I + A)^-1                                          (fp32, SIMT)
//   W^T  = K^T (T diag(beta gam rk))^T                         -> bf16 operand
//   U^T  = V^T (T diag(beta))^T          (T diag(beta) as a hi+lo bf16 pair)
//   Vn^T = U^T - S W^T                                         (into U's TMEM)
//   O1^T = S Q^T,  O2^T = Vn^T P^T,  P_ij = (q_i . k_j) e^{G_i - G_j} rk_j (j <= i)
//   o_i  = scale rq_i (gam_i O1_i + O2_i)
//   S   <- gam_last S + (Vn diag(d rk))^T K      (Vn diag(d rk) as a hi+lo pair)
//
// Every product is a tcgen05 MMA with M = 128 (the 128-wide head dimension on
// the M side), fp32 accumulators in TMEM.  K and Q enter the MMAs as the raw
// bf16 tiles TMA brought in; the L2 norms are folded into the fp32 diagonal
// factors, so only T-derived factors, W, S, P and Vn are rounded to bf16.  The
// two operands whose rounding reaches the state directly (T diag(beta) and
// Vn diag(d rk)) are split into hi + lo bf16 halves (~16 significant bits).
//
// TMEM columns (512 allocated):
//   [0,128) S fp32 | [128,192) Gram [K;Q] K^T | [192,256) W^T | [256,320) U^T -> Vn^T
//   [320,384) O1^T | [384,448) O2^T | [448,512) S as bf16 pairs (A operand)
//
// Masking: rows past the end of the sequence get beta = 0 and log g = 0, which
// makes their rows of T the identity and their rows of W, U and Vn exactly 0,
// so they never reach the state; their outputs are not stored.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <float.h>
#include <stdint.h>

#include "prefill.h"
#include "ptx.cuh"

namespace gdn {
namespace {

// ------------------------------------------------------------ shared memory map
constexpr uint32_t kKQBytes = 32768;   // [K dk0-63 | Q dk0-63 | K dk64-127 | Q dk64-127], 8 KB each
constexpr uint32_t kVBytes = 16384;    // [V dv0-63 | V dv64-127]
constexpr uint32_t OFF_KQ = 0;         // two buffers
constexpr uint32_t OFF_V = 2 * kKQBytes;
constexpr uint32_t OFF_P = OFF_V + 2 * kVBytes;  // P, 64 x 64 bf16 K-major (8 KB)
constexpr uint32_t OFF_U1 = OFF_P + 8192;        // phase-shared region (60 KB)
constexpr int kAStride = 68;                     // fp32 row stride of A and T (bank-conflict free)
constexpr uint32_t U1_A = 0;                     // A fp32 [64][68]
constexpr uint32_t U1_T = 17408;                 // T fp32 [64][68]
constexpr uint32_t U1_LW = 36864;                // T diag(beta gam rk), bf16 K-major (8 KB)
constexpr uint32_t U1_LUHI = 45056;              // T diag(beta) hi
constexpr uint32_t U1_LULO = 53248;              // T diag(beta) lo (first 4 KB double as solve scratch)
constexpr uint32_t U1_W = 0;                     // W as MN-major B operand, 128 rows x 128 B
constexpr uint32_t U1_VN = 0;                    // Vn^T bf16 K-major, 128 rows x 128 B
constexpr uint32_t U1_VDHI = 16384;              // (Vn diag(d rk))^T hi
constexpr uint32_t U1_VDLO = 32768;              // (Vn diag(d rk))^T lo
constexpr uint32_t U1_O = 0;                     // output staging [64][128] bf16
constexpr uint32_t kU1Bytes = 61440;
constexpr uint32_t OFF_VEC = OFF_U1 + kU1Bytes;  // per-row vectors, 64 floats each
constexpr int V_LG = 0, V_G = 1, V_BETA = 2, V_GAM = 3, V_D = 4, V_RK = 5, V_RQ = 6;
constexpr uint32_t kVecCount = 8;
constexpr uint32_t OFF_BAR = OFF_VEC + kVecCount * 64 * 4;
constexpr uint32_t kSmemUsed = OFF_BAR + 64;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // + alignment slack

static_assert(OFF_U1 % 1024 == 0 && (OFF_U1 + U1_LW) % 1024 == 0 && (OFF_U1 + U1_LUHI) % 1024 == 0 &&
                  (OFF_U1 + U1_LULO) % 1024 == 0 && (OFF_U1 + U1_VDHI) % 1024 == 0 &&
                  (OFF_U1 + U1_VDLO) % 1024 == 0,
              "UMMA operand blocks must be 1024-byte aligned");
static_assert(U1_T + 64 * kAStride * 4 <= U1_LW, "A/T overlap the L operands");
static_assert(U1_VDLO + 16384 <= kU1Bytes && U1_LULO + 8192 <= kU1Bytes, "phase region overflow");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// ------------------------------------------------------------ TMEM map
constexpr uint32_t TM_S = 0, TM_G = 128, TM_W = 192, TM_U = 256, TM_O1 = 320, TM_O2 = 384, TM_SB = 448;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kTileTxBytes = 2 * kKQBytes / 2 + kVBytes;  // K + Q + V = 48 KB per chunk
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;        // 200 ms per on-chip wait
constexpr int kThreads = 128;

constexpr int32_t kErrCu = 0x1, kErrIdx = 0x2, kErrTimeout = 0x4;

// ------------------------------------------------------------ small helpers
__device__ __forceinline__ int64_t load_index(const void* p, int dtype, int64_t i) {
  return dtype == kI64 ? reinterpret_cast<const int64_t*>(p)[i] : (int64_t) reinterpret_cast<const int32_t*>(p)[i];
}
__device__ __forceinline__ float load_real(const void* p, int dtype, int64_t i) {
  if (dtype == kF32) return reinterpret_cast<const float*>(p)[i];
  if (dtype == kBF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return __half2float(reinterpret_cast<const __half*>(p)[i]);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// hi = bf16(x), lo = bf16(x - hi): x ~= hi + lo to ~16 significant bits.
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}
__device__ __forceinline__ void set_error(int32_t* err, int32_t bit) { atomicOr(err, bit); }

// Read one 128-float row of a state slot (fp32 or bf16) into registers.
__device__ __forceinline__ void load_state_row(const void* base, int dtype, int64_t off, float (&row)[128]) {
  if (dtype == kF32) {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + off);
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      float4 x = __ldg(p + c);
      row[4 * c] = x.x; row[4 * c + 1] = x.y; row[4 * c + 2] = x.z; row[4 * c + 3] = x.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(base) + off);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      uint4 x = __ldg(p + c);
      uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&w[e]);
        float2 f = __bfloat1622float2(b);
        row[8 * c + 2 * e] = f.x; row[8 * c + 2 * e + 1] = f.y;
      }
    }
  }
}
__device__ __forceinline__ void store_state_chunk(void* base, int dtype, int64_t off, int c0, const float* v32) {
  if (dtype == kF32) {
    float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + off + c0);
#pragma unroll
    for (int c = 0; c < 8; ++c) p[c] = make_float4(v32[4 * c], v32[4 * c + 1], v32[4 * c + 2], v32[4 * c + 3]);
  } else {
    uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + off + c0);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      p[c] = make_uint4(pack_bf16(v32[8 * c], v32[8 * c + 1]), pack_bf16(v32[8 * c + 2], v32[8 * c + 3]),
                        pack_bf16(v32[8 * c + 4], v32[8 * c + 5]), pack_bf16(v32[8 * c + 6], v32[8 * c + 7]));
  }
}

// ------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kThreads, 1) gdn_prefill_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* vec = reinterpret_cast<float*>(sm + OFF_VEC);
  float* sLg = vec + V_LG * 64;
  float* sG = vec + V_G * 64;
  float* sBeta = vec + V_BETA * 64;
  float* sGam = vec + V_GAM * 64;
  float* sD = vec + V_D * 64;
  float* sRk = vec + V_RK * 64;
  float* sRq = vec + V_RQ * 64;
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + OFF_BAR);  // [2]
  uint64_t* bar_mma = bar_tma + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_tma + 3);
  uint8_t* u1 = sm + OFF_U1;
  float* sA = reinterpret_cast<float*>(u1 + U1_A);
  float* sT = reinterpret_cast<float*>(u1 + U1_T);
  float* sX = reinterpret_cast<float*>(u1 + U1_LULO);  // solve scratch (32 x 32 fp32)

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- the unit and its validation (uniform across the CTA)
  const int n = blockIdx.x / p.H;
  const int h = blockIdx.x - n * p.H;
  const int64_t bos = load_index(p.cu, p.cu_dtype, n);
  const int64_t eos = load_index(p.cu, p.cu_dtype, n + 1);
  if (bos < 0 || eos < bos || eos > p.T) {
    if (tid == 0) set_error(p.dev_err, kErrCu);
    return;
  }
  const int64_t slot = p.state_idx ? load_index(p.state_idx, p.idx_dtype, n) : (int64_t)n;
  if ((p.s_in && (slot < 0 || slot >= p.sin_slots)) || (p.s_out && (slot < 0 || slot >= p.sout_slots))) {
    if (tid == 0) set_error(p.dev_err, kErrIdx);
    return;
  }
  const int hq = h / (p.H / p.H_qk);
  const int hv = h / (p.H / p.H_v);
  const int64_t len = eos - bos;
  const int64_t sin_off = p.s_in ? slot * p.sin_slot + (int64_t)h * p.sin_head + (int64_t)tid * kHeadDim : 0;
  const int64_t sout_off = p.s_out ? slot * p.sout_slot + (int64_t)h * p.sout_head + (int64_t)tid * kHeadDim : 0;

  if (len == 0) {  // empty sequence: the final state is the initial state
    if (p.s_out) {
      float row[128];
      if (p.s_in) load_state_row(p.s_in, p.sin_dtype, sin_off, row);
      else {
#pragma unroll
        for (int j = 0; j < 128; ++j) row[j] = 0.f;
      }
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) store_state_chunk(p.s_out, p.sout_dtype, sout_off, c0, row + c0);
    }
    return;
  }
  const int nchunks = (int)((len + kChunk - 1) / kChunk);

  // ---- set-up: barriers, TMEM, first tile, initial state
  if (tid == 0) {
    mbar_init(&bar_tma[0], 1);
    mbar_init(&bar_tma[1], 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t trow = tmem + lane_base;  // this warp's lane quarter

  uint32_t tma_issued[2] = {0, 0};  // loads issued per buffer (thread 0 only)
  auto issue_tiles = [&](int c, int buf) {
    ++tma_issued[buf];
    const int t0 = (int)(bos + (int64_t)c * kChunk);
    uint8_t* kq = sm + OFF_KQ + buf * kKQBytes;
    uint8_t* vv = sm + OFF_V + buf * kVBytes;
    mbar_arrive_expect_tx(&bar_tma[buf], kTileTxBytes);
    tma_load_3d(kq + 0, &p.tm_k, &bar_tma[buf], 0, hq, t0);
    tma_load_3d(kq + 8192, &p.tm_q, &bar_tma[buf], 0, hq, t0);
    tma_load_3d(kq + 16384, &p.tm_k, &bar_tma[buf], 64, hq, t0);
    tma_load_3d(kq + 24576, &p.tm_q, &bar_tma[buf], 64, hq, t0);
    tma_load_3d(vv + 0, &p.tm_v, &bar_tma[buf], 0, hv, t0);
    tma_load_3d(vv + 8192, &p.tm_v, &bar_tma[buf], 64, hv, t0);
  };
  if (tid == 0) issue_tiles(0, 0);

  {  // initial state -> TMEM S (fp32) and S as bf16 pairs
    float row[128];
    if (p.s_in) load_state_row(p.s_in, p.sin_dtype, sin_off, row);
    else {
#pragma unroll
      for (int j = 0; j < 128; ++j) row[j] = 0.f;
    }
    uint32_t r[32];
#pragma unroll
    for (int c0 = 0; c0 < 128; c0 += 32) {
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(row[c0 + j]);
      tmem_st32(trow + TM_S + c0, r);
    }
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 32) {
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = pack_bf16(row[2 * (c0 + j)], row[2 * (c0 + j) + 1]);
      tmem_st32(trow + TM_SB + c0, r);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const float eps = 1e-6f;
  uint32_t mma_phase = 0;
  bool failed = false;

  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    const int64_t t0 = bos + (int64_t)c * kChunk;
    const int nvalid = (eos - t0 < kChunk) ? (int)(eos - t0) : kChunk;
    const bool last = (c + 1 == nchunks);
    uint8_t* kq = sm + OFF_KQ + buf * kKQBytes;
    uint8_t* vv = sm + OFF_V + buf * kVBytes;
    const uint32_t kq_a = smem_u32(kq), v_a = smem_u32(vv);

    if (tid == 0 && !last) issue_tiles(c + 1, buf ^ 1);
    {
      bool ok = mbar_wait(&bar_tma[buf], (uint32_t)((c >> 1) & 1), kWaitLimitNs);
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }

    // ---- Gram [K;Q] K^T (M = 128: rows 0-63 k_i, 64-127 q_i; N = 64)
    if (tid == 0) {
      const uint32_t id = idesc_bf16_f32(128, 64, 0, 0, 0);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint64_t d = sdesc_sw128(kq_a + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024);
        mma_ss(tmem + TM_G, d, d, id, s > 0);
      }
      mma_commit(bar_mma);
    }
    // ---- gates (warps 0-1) and q norms (warps 2-3)
    if (warp < 2) {
      const int i = tid;
      float lg = 0.f, bt = 0.f;
      if (i < nvalid) {
        const int64_t t = t0 + i;
        if (p.g) lg = __logf(fmaxf(load_real(p.g, p.g_dtype, t * p.g_st + (int64_t)h * p.g_sh), FLT_MIN));
        bt = p.beta ? load_real(p.beta, p.b_dtype, t * p.b_st + (int64_t)h * p.b_sh) : 1.f;
      }
      float x = lg;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      sLg[i] = x;
      sBeta[i] = bt;
    } else {
      const int i = tid - 64;
      float ss = 0.f;
      if (p.l2norm) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint8_t* row = kq + 8192 + half * 16384 + i * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint4 w = *reinterpret_cast<const uint4*>(row + (((k + i) & 7) << 4));
            uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&ws[e]));
              ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
            }
          }
        }
      }
      sRq[i] = p.l2norm ? rsqrtf(ss + eps) : 1.f;
    }
    __syncthreads();

    float gram[64];  // warps 0-1: row i of K K^T; warps 2-3: row i of Q K^T
    {
      if (warp < 2) sG[tid] = sLg[tid] + (tid >= 32 ? sLg[31] : 0.f);
      bool ok = mbar_wait(bar_mma, mma_phase, kWaitLimitNs);
      mma_phase ^= 1;
      tc_fence_after();
      uint32_t r[32];
      tmem_ld32(trow + TM_G, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) gram[j] = __uint_as_float(r[j]);
      tmem_ld32(trow + TM_G + 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) gram[32 + j] = __uint_as_float(r[j]);
      if (warp < 2) {
        const int i = tid;
        float kk = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) kk = (j == i) ? gram[j] : kk;
        sRk[i] = p.l2norm ? rsqrtf(kk + eps) : 1.f;
        sGam[i] = __expf(sG[i]);
      }
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    if (warp < 2) {  // A rows (fp32) and the decay vector d
      const int i = tid;
      const float Gi = sG[i], Glast = sG[63];
      sD[i] = __expf(Glast - Gi);
      const float bi = sBeta[i] * sRk[i];
      float* arow = sA + i * kAStride;
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        float a[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int jj = j + e;
          a[e] = (jj < i) ? bi * __expf(Gi - sG[jj]) * sRk[jj] * gram[jj] : 0.f;
        }
        *reinterpret_cast<float4*>(arow + j) = make_float4(a[0], a[1], a[2], a[3]);
      }
    } else {  // P rows (bf16, K-major)
      const int i = tid - 64;
      const float Gi = sG[i];
      uint8_t* sP = sm + OFF_P;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j0 = ch * 8 + 2 * e, j1 = j0 + 1;
          const float p0 = (j0 <= i) ? gram[j0] * __expf(Gi - sG[j0]) * sRk[j0] : 0.f;
          const float p1 = (j1 <= i) ? gram[j1] * __expf(Gi - sG[j1]) * sRk[j1] : 0.f;
          w[e] = pack_bf16(p0, p1);
        }
        *reinterpret_cast<uint4*>(sP + sw128_chunk(i, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    __syncthreads();

    // ---- T = (I + A)^-1 by 32 x 32 blocks: diagonal blocks by column substitution,
    //      then T21 = -T22 (A21 T11).
    if (tid < 64) {
      const int base = (tid >> 5) * 32;
      const int m = tid & 31;
      float t[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float* arow = sA + (base + i) * kAStride + base;
        float acc = (i == m) ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < i; ++j) acc = fmaf(-arow[j], t[j], acc);
        t[i] = acc;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) sT[(base + i) * kAStride + base + m] = t[i];
    }
    __syncthreads();
    {
      const int cc = tid & 31, r0 = (tid >> 5) * 8;
#pragma unroll
      for (int r = r0; r < r0 + 8; ++r) {
        const float* arow = sA + (32 + r) * kAStride;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) acc = fmaf(arow[k], sT[k * kAStride + cc], acc);
        sX[r * 32 + cc] = acc;
      }
    }
    __syncthreads();
    {
      const int cc = tid & 31, r0 = (tid >> 5) * 8;
#pragma unroll
      for (int r = r0; r < r0 + 8; ++r) {
        const float* trow22 = sT + (32 + r) * kAStride + 32;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) acc = fmaf(trow22[k], sX[k * 32 + cc], acc);
        sT[(32 + r) * kAStride + cc] = -acc;
      }
    }
    __syncthreads();

    // ---- operands T diag(beta gam rk) (bf16) and T diag(beta) (hi + lo), K-major rows i
    {
      const int i = tid >> 1, hf = tid & 1;
      uint8_t* lw = u1 + U1_LW;
      uint8_t* luh = u1 + U1_LUHI;
      uint8_t* lul = u1 + U1_LULO;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int ch = hf * 4 + q4;
        uint32_t ww[4], wh[4], wl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j0 = ch * 8 + 2 * e, j1 = j0 + 1;
          const bool upper = (i < 32) && (j0 >= 32);
          const float t0v = upper ? 0.f : sT[i * kAStride + j0];
          const float t1v = upper ? 0.f : sT[i * kAStride + j1];
          const float b0 = sBeta[j0], b1 = sBeta[j1];
          ww[e] = pack_bf16(t0v * b0 * sGam[j0] * sRk[j0], t1v * b1 * sGam[j1] * sRk[j1]);
          split_bf16(t0v * b0, t1v * b1, wh[e], wl[e]);
        }
        const uint32_t o = sw128_chunk(i, ch);
        *reinterpret_cast<uint4*>(lw + o) = make_uint4(ww[0], ww[1], ww[2], ww[3]);
        *reinterpret_cast<uint4*>(luh + o) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4*>(lul + o) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- W^T = K^T (T diag(beta gam rk))^T and U^T = V^T (T diag(beta))^T  (M = 128, N = 64, K = 64)
    if (tid == 0) {
      const uint32_t id = idesc_bf16_f32(128, 64, 1, 0, 0);
      const uint32_t lw = smem_u32(u1 + U1_LW), luh = smem_u32(u1 + U1_LUHI), lul = smem_u32(u1 + U1_LULO);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma_ss(tmem + TM_W, sdesc_sw128(kq_a + s * 2048, 16384, 1024), sdesc_sw128(lw + s * 32, 16, 1024), id, s > 0);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma_ss(tmem + TM_U, sdesc_sw128(v_a + s * 2048, 8192, 1024), sdesc_sw128(luh + s * 32, 16, 1024), id, s > 0);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma_ss(tmem + TM_U, sdesc_sw128(v_a + s * 2048, 8192, 1024), sdesc_sw128(lul + s * 32, 16, 1024), id, 1);
      mma_commit(bar_mma);
    }
    {
      bool ok = mbar_wait(bar_mma, mma_phase, kWaitLimitNs);
      mma_phase ^= 1;
      tc_fence_after();
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    // ---- W^T row dk -> W as the MN-major B operand (row dk holds the 64 tokens)
    {
      uint32_t r[32], w[32];
      uint8_t* sw = u1 + U1_W;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        tmem_ld32(trow + TM_W + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          *reinterpret_cast<uint4*>(sw + sw128_chunk(tid, c0 / 8 + q4)) =
              make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- Vn^T = U^T - S W^T and O1^T = S Q^T  (A = S as bf16 from TMEM, K = 128)
    if (tid == 0) {
      const uint32_t idx = idesc_bf16_f32(128, 64, 0, 1, 1);
      const uint32_t ido = idesc_bf16_f32(128, 64, 0, 0, 0);
      const uint32_t sw = smem_u32(u1 + U1_W);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        mma_ts(tmem + TM_U, tmem + TM_SB + s * 8, sdesc_sw128(sw + s * 2048, 8192, 1024), idx, 1);
        mma_ts(tmem + TM_O1, tmem + TM_SB + s * 8,
               sdesc_sw128(kq_a + 8192 + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024), ido, s > 0);
      }
      mma_commit(bar_mma);
    }
    {
      bool ok = mbar_wait(bar_mma, mma_phase, kWaitLimitNs);
      mma_phase ^= 1;
      tc_fence_after();
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    // ---- epilogue 1 (thread = value row v): Vn^T as bf16, (Vn diag(d rk))^T as hi + lo,
    //      and S <- gam_last S ahead of the state-update MMA.
    {
      uint32_t r[32];
      uint8_t* svn = u1 + U1_VN;
      uint8_t* svh = u1 + U1_VDHI;
      uint8_t* svl = u1 + U1_VDLO;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        tmem_ld32(trow + TM_U + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t wn[4], wh[4], wl[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 8 * q4 + 2 * e;
            const float a = __uint_as_float(r[j]), b = __uint_as_float(r[j + 1]);
            wn[e] = pack_bf16(a, b);
            const int jj = c0 + j;
            split_bf16(a * sD[jj] * sRk[jj], b * sD[jj + 1] * sRk[jj + 1], wh[e], wl[e]);
          }
          const uint32_t o = sw128_chunk(tid, c0 / 8 + q4);
          *reinterpret_cast<uint4*>(svn + o) = make_uint4(wn[0], wn[1], wn[2], wn[3]);
          *reinterpret_cast<uint4*>(svh + o) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
          *reinterpret_cast<uint4*>(svl + o) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
      }
      const float gl = sGam[63];
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        tmem_ld32(trow + TM_S + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * gl);
        tmem_st32(trow + TM_S + c0, r);
      }
      tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- O2^T = Vn^T P^T (K = 64) and S += (Vn diag(d rk))^T K  (hi, then lo; N = 128)
    if (tid == 0) {
      const uint32_t ido = idesc_bf16_f32(128, 64, 0, 0, 0);
      const uint32_t ids = idesc_bf16_f32(128, 128, 0, 1, 0);
      const uint32_t svn = smem_u32(u1 + U1_VN), svh = smem_u32(u1 + U1_VDHI), svl = smem_u32(u1 + U1_VDLO);
      const uint32_t sp = smem_u32(sm + OFF_P);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma_ss(tmem + TM_O2, sdesc_sw128(svn + s * 32, 16, 1024), sdesc_sw128(sp + s * 32, 16, 1024), ido, s > 0);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma_ss(tmem + TM_S, sdesc_sw128(svh + s * 32, 16, 1024), sdesc_sw128(kq_a + s * 2048, 16384, 1024), ids, 1);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma_ss(tmem + TM_S, sdesc_sw128(svl + s * 32, 16, 1024), sdesc_sw128(kq_a + s * 2048, 16384, 1024), ids, 1);
      mma_commit(bar_mma);
    }
    {
      bool ok = mbar_wait(bar_mma, mma_phase, kWaitLimitNs);
      mma_phase ^= 1;
      tc_fence_after();
      if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    // ---- epilogue 2: S -> bf16 copy for the next chunk (or the final state), output tile
    {
      uint32_t r[32];
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        tmem_ld32(trow + TM_S + c0, r);
        tmem_ld_wait();
        if (last) {
          if (p.s_out) {
            float v32[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v32[j] = __uint_as_float(r[j]);
            store_state_chunk(p.s_out, p.sout_dtype, sout_off, c0, v32);
          }
        } else {
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) w[j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
          asm volatile(
              "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
                  trow + TM_SB + c0 / 2),
              "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]),
              "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
              : "memory");
        }
      }
      __nv_bfloat16* so = reinterpret_cast<__nv_bfloat16*>(u1 + U1_O);
      uint32_t r2[32];
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        tmem_ld32(trow + TM_O1 + c0, r);
        tmem_ld32(trow + TM_O2 + c0, r2);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int i = c0 + j;
          const float o = p.scale * sRq[i] * fmaf(sGam[i], __uint_as_float(r[j]), __uint_as_float(r2[j]));
          so[i * 128 + tid] = __float2bfloat16_rn(o);
        }
      }
      tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    {  // coalesced store of the valid output rows
      const uint4* so = reinterpret_cast<const uint4*>(u1 + U1_O);
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int idx = tid + k * kThreads;
        const int row = idx >> 4, ch = idx & 15;
        if (row < nvalid) {
          uint4* dst = reinterpret_cast<uint4*>(out + (t0 + row) * p.o_st + (int64_t)h * p.o_sh) + ch;
          *dst = so[row * 16 + ch];
        }
      }
    }
    __syncthreads();  // the staging area is reused by the next chunk
  }

  if (failed) {
    if (tid == 0) {
      set_error(p.dev_err, kErrTimeout);
      // let the last tile load of each buffer land before the CTA's shared memory goes away
      for (int b = 0; b < 2; ++b)
        if (tma_issued[b]) mbar_wait(&bar_tma[b], (tma_issued[b] - 1) & 1, kWaitLimitNs);
    }
    __syncthreads();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

size_t prefill_smem_bytes() { return kSmemBytes; }

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(gdn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int64_t units = (int64_t)p.N * p.H;
  if (units == 0) return cudaSuccess;
  gdn_prefill_kernel<<<(unsigned)units, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
