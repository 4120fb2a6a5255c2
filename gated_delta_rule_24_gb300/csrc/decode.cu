// One Gated Delta Rule decode step for sm_103a: for each batch row b and sab head h the
// state slot S (V-major 128 x 128: row = value index, column = key index) takes one
// token and is updated in place,
//
//   S' = g S (I - beta k k^T) + beta v k^T = g S + delta k^T,   delta = beta (v - g S k)
//   o  = scale S' q = scale (g S q + delta (k . q))
//
// (the token recurrence of flashinfer.cudnn.cudnn_chunk_gated_delta_rule, Parameters,
// with one token per sequence; k and q are L2-normalised first when asked).  S is read
// once and written once, so the step is bound by HBM bandwidth.  A CTA of 128 threads
// takes a state in four groups of 32 rows, four threads per row and 32 columns per thread.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <float.h>
#include <stdint.h>

#include "decode.h"
#include "prefill.h"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int kDecRows = 32;                // state rows per row group
constexpr int kDecThreads = 4 * kDecRows;   // four threads per row
constexpr int kDecParts = kHeadDim / kDecRows;
constexpr int32_t kErrIdx = 0x2, kErrTimeout = 0x4;
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // every wait is bounded

__device__ __forceinline__ int64_t idx_at(const void* p, int dtype, int64_t i) {
  return dtype == kI64 ? reinterpret_cast<const int64_t*>(p)[i] : (int64_t)reinterpret_cast<const int32_t*>(p)[i];
}
// q/k/v element (bf16, or fp16 when f16)
__device__ __forceinline__ float in16(const void* p, int64_t i, bool f16) {
  return f16 ? __half2float(reinterpret_cast<const __half*>(p)[i])
             : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
}
__device__ __forceinline__ float real_at(const void* p, int dtype, int64_t i) {
  if (dtype == kF32) return reinterpret_cast<const float*>(p)[i];
  if (dtype == kBF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return __half2float(reinterpret_cast<const __half*>(p)[i]);
}

// The thread's 32 columns are the 16-byte chunks qd, qd + 4, ..., qd + 28 of its row (four
// consecutive threads cover 64 contiguous bytes per load).
template <int SDT>
__device__ __forceinline__ void load_row32(const void* row, int qd, float (&s)[32]) {
  if (SDT != 0) {
    const uint4* r = reinterpret_cast<const uint4*>(row);  // 8 bf16 per 16-byte chunk
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 c = r[qd + 4 * j];
      const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (SDT == 2) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          s[8 * j + 2 * e] = f.x;
          s[8 * j + 2 * e + 1] = f.y;
        } else {
          s[8 * j + 2 * e] = __uint_as_float(w[e] << 16);
          s[8 * j + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
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
template <int SDT>
__device__ __forceinline__ int col_of(int qd, int e) {
  return SDT != 0 ? 8 * (qd + 4 * (e >> 3)) + (e & 7) : 4 * (qd + 4 * (e >> 2)) + (e & 3);
}
template <int SDT>
__device__ __forceinline__ void store_row32(void* row, int qd, const float (&s)[32]) {
  if (SDT != 0) {
    uint4* r = reinterpret_cast<uint4*>(row);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (SDT == 2) {
          __half2 h = __floats2half2_rn(s[8 * j + 2 * e], s[8 * j + 2 * e + 1]);
          w[e] = *reinterpret_cast<uint32_t*>(&h);
        } else {
          __nv_bfloat162 h = __floats2bfloat162_rn(s[8 * j + 2 * e], s[8 * j + 2 * e + 1]);
          w[e] = *reinterpret_cast<uint32_t*>(&h);
        }
      }
      r[qd + 4 * j] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    float4* r = reinterpret_cast<float4*>(row);
#pragma unroll
    for (int j = 0; j < 8; ++j) r[qd + 4 * j] = make_float4(s[4 * j], s[4 * j + 1], s[4 * j + 2], s[4 * j + 3]);
  }
}

// Persistent CTAs walk the work items (b, h) -- one state each -- with a ring of
// shared-memory stages: thread 0 keeps bulk copies of the next items' whole states in
// flight (no registers held), and the per-item inputs (k, q, v, g, beta and their norms)
// are fetched once per 64 KB (bf16: 32 KB) state rather than once per row group.
template <int SDT>
__host__ __device__ constexpr int dec_stages() { return 2; }  // three bf16 (two f32) CTAs per SM
constexpr int kMaxDecStages = 2;

struct DecodeSmem {
  float kh[128], qh[128];
  float red[3][4];
  uint64_t full[kMaxDecStages];
};

__device__ __forceinline__ bool item_slot(const DecodeParams& p, int64_t item, int64_t& slot, int& b, int& h) {
  b = (int)(item / p.H);
  h = (int)(item - (int64_t)b * p.H);
  slot = p.state_idx ? idx_at(p.state_idx, p.idx_dtype, b) : (int64_t)b;
  return slot >= 0 && slot < p.st_slots;
}

template <int SDT>
__global__ void __launch_bounds__(kDecThreads) gdn_decode_kernel(const __grid_constant__ DecodeParams p,
                                                                 int64_t n_items) {
  static_assert(kDecThreads == kHeadDim, "one thread per key element in the prologue");
  constexpr uint32_t kRowBytes = kHeadDim * (SDT != 0 ? 2 : 4);
  constexpr uint32_t kStageBytes = kHeadDim * kRowBytes;  // one whole state
  constexpr int kStages = dec_stages<SDT>();
  extern __shared__ __align__(128) uint8_t dsm[];
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(dsm + kStages * kStageBytes);
  const int t = threadIdx.x, qd = t & 3;
  if (t == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(&sm.full[st], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto state_ptr = [&](int64_t slot, int h) -> char* {
    return reinterpret_cast<char*>(p.state) + (slot * p.st_slot + (int64_t)h * p.st_head) * (SDT != 0 ? 2 : 4);
  };
  // local item j of this CTA goes to stage j % kStages (invalid items still advance the
  // stage's phase, with an arrival and no copy)
  auto issue = [&](int64_t j) {
    const int64_t item = blockIdx.x + j * gridDim.x;
    if (item >= n_items) return;
    int64_t slot;
    int b, h;
    const int st = (int)(j % kStages);
    if (!item_slot(p, item, slot, b, h)) {
      mbar_arrive(&sm.full[st]);
      return;
    }
    mbar_arrive_expect_tx(&sm.full[st], kStageBytes);
    bulk_load(dsm + st * kStageBytes, state_ptr(slot, h), kStageBytes, &sm.full[st]);
  };
  if (t == 0)
    for (int j = 0; j < kStages; ++j) issue(j);
  bool ok = true;
  int64_t j = 0;
  for (; ok; ++j) {
    const int64_t item = blockIdx.x + j * gridDim.x;
    if (item >= n_items) break;
    int64_t slot;
    int b, h;
    const bool valid = item_slot(p, item, slot, b, h);
    const int st = (int)(j % kStages);
    if (!valid) {  // uniform over the CTA; nothing was loaded for it
      if (t == 0) {
        atomicOr(p.dev_err, kErrIdx);
        issue(j + kStages);
      }
      continue;
    }
    const int hq = h / (p.H / p.H_qk), hv = h / (p.H / p.H_v);
    const bool f16 = p.in_f16 != 0;
    const float kx = in16(p.k, b * p.k_sb + (int64_t)hq * p.k_sh + t, f16);
    const float qx = in16(p.q, b * p.q_sb + (int64_t)hq * p.q_sh + t, f16);
    const int64_t vrow = b * p.v_sb + (int64_t)hv * p.v_sh;
    float vr[kDecParts];
#pragma unroll
    for (int pt = 0; pt < kDecParts; ++pt) vr[pt] = in16(p.v, vrow + pt * kDecRows + (t >> 2), f16);
    float g = 1.f, beta = 1.f;
    if (p.g) g = fminf(fmaxf(real_at(p.g, p.g_dtype, b * p.g_sb + (int64_t)h * p.g_sh), FLT_MIN), 1.f);
    if (p.beta) beta = real_at(p.beta, p.b_dtype, b * p.b_sb + (int64_t)h * p.b_sh);
    float a = kx * kx, c = qx * qx, d = kx * qx;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      c += __shfl_xor_sync(0xffffffffu, c, o);
      d += __shfl_xor_sync(0xffffffffu, d, o);
    }
    if ((t & 31) == 0) { sm.red[0][t >> 5] = a; sm.red[1][t >> 5] = c; sm.red[2][t >> 5] = d; }
    sm.kh[t] = kx;
    sm.qh[t] = qx;
    const bool w = mbar_wait(&sm.full[st], (uint32_t)((j / kStages) & 1), kWaitLimitNs);
    ok = __syncthreads_and(w);
    if (!ok) break;  // j stays the first item whose copy may be outstanding
    const float kk = sm.red[0][0] + sm.red[0][1] + sm.red[0][2] + sm.red[0][3];
    const float qq = sm.red[1][0] + sm.red[1][1] + sm.red[1][2] + sm.red[1][3];
    const float kq_raw = sm.red[2][0] + sm.red[2][1] + sm.red[2][2] + sm.red[2][3];
    const float rk = p.l2norm ? rsqrtf(kk + 1e-6f) : 1.f, rq = p.l2norm ? rsqrtf(qq + 1e-6f) : 1.f;
    char* sbase = state_ptr(slot, h);
#pragma unroll 1
    for (int pt = 0; pt < kDecParts; ++pt) {
      const int rr = pt * kDecRows + (t >> 2);
      float s[32];
      load_row32<SDT>(dsm + st * kStageBytes + rr * kRowBytes, qd, s);
      float u = 0.f, wq = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int cc = col_of<SDT>(qd, e);
        u = fmaf(s[e], sm.kh[cc], u);
        wq = fmaf(s[e], sm.qh[cc], wq);
      }
      u += __shfl_xor_sync(0xffffffffu, u, 1);
      wq += __shfl_xor_sync(0xffffffffu, wq, 1);
      u += __shfl_xor_sync(0xffffffffu, u, 2);
      wq += __shfl_xor_sync(0xffffffffu, wq, 2);
      u *= rk;
      wq *= rq;
      float vv = vr[0];
#pragma unroll
      for (int q2 = 1; q2 < kDecParts; ++q2) vv = (pt == q2) ? vr[q2] : vv;
      const float delta = beta * (vv - g * u);  // beta (v - g S k^)
      if (qd == 0) {
        const float o = p.scale * (g * wq + delta * (kq_raw * rk * rq));
        const int64_t oi = b * p.o_sb + (int64_t)h * p.o_sh + rr;
        if (f16) reinterpret_cast<__half*>(p.out)[oi] = __float2half_rn(o);
        else reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
      }
      const float dk = delta * rk;  // S' = g S + delta k^T with k^ = rk k
#pragma unroll
      for (int e = 0; e < 32; ++e) s[e] = fmaf(g, s[e], dk * sm.kh[col_of<SDT>(qd, e)]);
      store_row32<SDT>(sbase + rr * kRowBytes, qd, s);
    }
    // every row of the stage has been read (and the vectors are no longer needed): the
    // stage takes the item kStages ahead
    __syncthreads();
    if (t == 0) issue(j + kStages);
  }
  if (!ok && t == 0) {
    atomicOr(p.dev_err, kErrTimeout);
    // let the copies already issued (items j .. j + kStages - 1) land before the CTA's
    // shared memory goes away
    for (int64_t jj = j; jj < j + kStages; ++jj) {
      const int64_t item = blockIdx.x + jj * gridDim.x;
      int64_t slot;
      int b, h;
      if (item < n_items && item_slot(p, item, slot, b, h))
        mbar_wait(&sm.full[jj % kStages], (uint32_t)((jj / kStages) & 1), kWaitLimitNs);
    }
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  const int64_t items = (int64_t)p.B * p.H;
  if (items <= 0) return cudaSuccess;
  static thread_local int configured = -1, configured_gen = -1, sms = 0, per_sm[3] = {0, 0, 0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int gen = launch_config_generation();
  const size_t smem_bf = dec_stages<1>() * kHeadDim * kHeadDim * 2 + sizeof(DecodeSmem);  // 16-bit states
  const size_t smem_f32 = dec_stages<0>() * kHeadDim * kHeadDim * 4 + sizeof(DecodeSmem);
  if (configured != dev || configured_gen != gen) {
    e = cudaFuncSetAttribute(gdn_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bf);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gdn_decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bf);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gdn_decode_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_f32);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // resident CTAs per SM for each state type, queried once so that a launch makes no
    // runtime call but the launch itself (and so can be captured into a CUDA graph)
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[0], gdn_decode_kernel<0>, kDecThreads, smem_f32);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[1], gdn_decode_kernel<1>, kDecThreads, smem_bf);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[2], gdn_decode_kernel<2>, kDecThreads, smem_bf);
    if (e != cudaSuccess) return e;
    configured = dev;
    configured_gen = gen;
  }
  const int sdt = p.st_dtype == kBF16 ? 1 : (p.st_dtype == kF16 ? 2 : 0);
  const size_t smem = sdt ? smem_bf : smem_f32;
  const int64_t cap = (int64_t)sms * (per_sm[sdt] > 0 ? per_sm[sdt] : 1);
  const unsigned grid = (unsigned)(items < cap ? items : cap);
  if (sdt == 1) gdn_decode_kernel<1><<<grid, kDecThreads, smem, stream>>>(p, items);
  else if (sdt == 2) gdn_decode_kernel<2><<<grid, kDecThreads, smem, stream>>>(p, items);
  else gdn_decode_kernel<0><<<grid, kDecThreads, smem, stream>>>(p, items);
  return cudaGetLastError();
}

}  // namespace gdn
