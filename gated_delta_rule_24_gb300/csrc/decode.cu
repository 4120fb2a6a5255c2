// One Gated Delta Rule decode step for sm_103a: for each batch row b and sab head h the
// state slot S (V-major 128 x 128: row = value index, column = key index) takes one
// token and is updated in place,
//
//   S' = g S (I - beta k k^T) + beta v k^T = g S + delta k^T,   delta = beta (v - g S k)
//   o  = scale S' q = scale (g S q + delta (k . q))
//
// (the token recurrence of flashinfer.cudnn.cudnn_chunk_gated_delta_rule, Parameters,
// with one token per sequence; k and q are L2-normalised first when asked).  S is read
// once and written once, so the step is bound by HBM bandwidth: four CTAs of 128 threads
// per (b, h), each taking 32 state rows with four threads per row and 32 columns per
// thread in registers (small CTAs keep several resident per SM for memory parallelism).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <float.h>
#include <stdint.h>

#include "decode.h"
#include "prefill.h"

namespace gdn {
namespace {

constexpr int kDecRows = 32;                // state rows per CTA
constexpr int kDecThreads = 4 * kDecRows;   // four threads per row
constexpr int kDecParts = kHeadDim / kDecRows;
constexpr int32_t kErrIdx = 0x2;

__device__ __forceinline__ int64_t idx_at(const void* p, int dtype, int64_t i) {
  return dtype == kI64 ? reinterpret_cast<const int64_t*>(p)[i] : (int64_t)reinterpret_cast<const int32_t*>(p)[i];
}
__device__ __forceinline__ float real_at(const void* p, int dtype, int64_t i) {
  if (dtype == kF32) return reinterpret_cast<const float*>(p)[i];
  if (dtype == kBF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return __half2float(reinterpret_cast<const __half*>(p)[i]);
}

// The thread's 32 columns are the 16-byte chunks qd, qd + 4, ..., qd + 28 of its row (four
// consecutive threads cover 64 contiguous bytes per load).
template <bool BF16>
__device__ __forceinline__ void load_row32(const void* row, int qd, float (&s)[32]) {
  if (BF16) {
    const uint4* r = reinterpret_cast<const uint4*>(row);  // 8 bf16 per 16-byte chunk
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 c = r[qd + 4 * j];
      const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s[8 * j + 2 * e] = __uint_as_float(w[e] << 16);
        s[8 * j + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
      }
    }
  } else {
    const float4* r = reinterpret_cast<const float4*>(row);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 c = r[qd + 4 * j];
      s[4 * j] = c.x; s[4 * j + 1] = c.y; s[4 * j + 2] = c.z; s[4 * j + 3] = c.w;
    }
  }
}
// Column of element e of the thread's 32 (see load_row32).
template <bool BF16>
__device__ __forceinline__ int col_of(int qd, int e) {
  return BF16 ? 8 * (qd + 4 * (e >> 3)) + (e & 7) : 4 * (qd + 4 * (e >> 2)) + (e & 3);
}
template <bool BF16>
__device__ __forceinline__ void store_row32(void* row, int qd, const float (&s)[32]) {
  if (BF16) {
    uint4* r = reinterpret_cast<uint4*>(row);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 h = __floats2bfloat162_rn(s[8 * j + 2 * e], s[8 * j + 2 * e + 1]);
        w[e] = *reinterpret_cast<uint32_t*>(&h);
      }
      r[qd + 4 * j] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    float4* r = reinterpret_cast<float4*>(row);
#pragma unroll
    for (int j = 0; j < 8; ++j) r[qd + 4 * j] = make_float4(s[4 * j], s[4 * j + 1], s[4 * j + 2], s[4 * j + 3]);
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kDecThreads) gdn_decode_kernel(const __grid_constant__ DecodeParams p) {
  static_assert(kDecThreads == kHeadDim, "one thread per key element in the prologue");
  __shared__ float kh[128], qh[128];  // key and query (raw; the norm factors are applied after)
  __shared__ float red[3][4];         // |k|^2, |q|^2, k.q per warp
  const int bh = blockIdx.x / kDecParts, part = blockIdx.x - bh * kDecParts;
  const int b = bh / p.H, h = bh - b * p.H;
  const int t = threadIdx.x, r = part * kDecRows + (t >> 2), qd = t & 3;
  const int hq = h / (p.H / p.H_qk), hv = h / (p.H / p.H_v);
  const int64_t slot = p.state_idx ? idx_at(p.state_idx, p.idx_dtype, b) : (int64_t)b;
  if (slot < 0 || slot >= p.st_slots) {  // uniform over the CTA
    if (t == 0) atomicOr(p.dev_err, kErrIdx);
    return;
  }
  // the state row first: its load is the long one
  char* row = reinterpret_cast<char*>(p.state) +
              (slot * p.st_slot + (int64_t)h * p.st_head + (int64_t)r * kHeadDim) * (BF16 ? 2 : 4);
  float s[32];
  load_row32<BF16>(row, qd, s);
  float g = 1.f, beta = 1.f;
  if (p.g) g = fminf(fmaxf(real_at(p.g, p.g_dtype, b * p.g_sb + (int64_t)h * p.g_sh), FLT_MIN), 1.f);
  if (p.beta) beta = real_at(p.beta, p.b_dtype, b * p.b_sb + (int64_t)h * p.b_sh);
  const float vr = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.v)[b * p.v_sb + (int64_t)hv * p.v_sh + r]);
  {
    const float kx = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.k)[b * p.k_sb + (int64_t)hq * p.k_sh + t]);
    const float qx = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.q)[b * p.q_sb + (int64_t)hq * p.q_sh + t]);
    float a = kx * kx, c = qx * qx, d = kx * qx;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      c += __shfl_xor_sync(0xffffffffu, c, o);
      d += __shfl_xor_sync(0xffffffffu, d, o);
    }
    if ((t & 31) == 0) { red[0][t >> 5] = a; red[1][t >> 5] = c; red[2][t >> 5] = d; }
    kh[t] = kx;
    qh[t] = qx;
  }
  __syncthreads();
  const float kk = red[0][0] + red[0][1] + red[0][2] + red[0][3];
  const float qq = red[1][0] + red[1][1] + red[1][2] + red[1][3];
  const float kq_raw = red[2][0] + red[2][1] + red[2][2] + red[2][3];
  const float rk = p.l2norm ? rsqrtf(kk + 1e-6f) : 1.f, rq = p.l2norm ? rsqrtf(qq + 1e-6f) : 1.f;
  // u = S k, w = S q over this thread's columns, then across the row's four threads
  float u = 0.f, w = 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const int c = col_of<BF16>(qd, e);
    u = fmaf(s[e], kh[c], u);
    w = fmaf(s[e], qh[c], w);
  }
  u += __shfl_xor_sync(0xffffffffu, u, 1);
  w += __shfl_xor_sync(0xffffffffu, w, 1);
  u += __shfl_xor_sync(0xffffffffu, u, 2);
  w += __shfl_xor_sync(0xffffffffu, w, 2);
  u *= rk;
  w *= rq;
  const float delta = beta * (vr - g * u);  // beta (v - g S k^)
  if (qd == 0) {
    const float o = p.scale * (g * w + delta * (kq_raw * rk * rq));
    reinterpret_cast<__nv_bfloat16*>(p.out)[b * p.o_sb + (int64_t)h * p.o_sh + r] = __float2bfloat16_rn(o);
  }
  const float dk = delta * rk;  // S' = g S + delta k^T with k^ = rk k
#pragma unroll
  for (int e = 0; e < 32; ++e) s[e] = fmaf(g, s[e], dk * kh[col_of<BF16>(qd, e)]);
  store_row32<BF16>(row, qd, s);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  const int64_t ctas = (int64_t)p.B * p.H * kDecParts;
  if (ctas <= 0) return cudaSuccess;
  if (p.st_dtype == kBF16) gdn_decode_kernel<true><<<(unsigned)ctas, kDecThreads, 0, stream>>>(p);
  else gdn_decode_kernel<false><<<(unsigned)ctas, kDecThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
