// Chunked Gated Delta Rule prefill for sm_103a: a persistent, warp-specialised
// kernel.  Each CTA walks the (sequence, sab head) units u = blockIdx.x,
// blockIdx.x + gridDim.x, ... and, inside a unit, its 64-token chunks in order.
//
// For a chunk (rows i, j = 0..63; raw 16-bit tiles K, Q of the q/k head and V of the
// v head; gates g, beta; S the Dv x Dk fp32 state entering the chunk, row = value
// index) the chunk-parallel delta rule (Yang et al., "Parallelizing Linear
// Transformers with the Delta Rule over Sequence Length"; gated as in "Gated Delta
// Networks") is evaluated as
//
//   G = cumsum(log g),  gam_i = e^{G_i},  d_j = e^{G_last - G_j}
//   rk_i, rq_i = 1/sqrt(|k_i|^2 + 1e-6), 1/sqrt(|q_i|^2 + 1e-6)   (1 without L2 norm)
//   A_ij = beta_i e^{G_i - G_j} rk_i rk_j (k_i . k_j)   (j < i),   T = (I + A)^-1
//   W    = T diag(beta gam rk) K          U = T diag(beta) V
//   P_ij = (q_i . k_j) e^{G_i - G_j} rk_j   (j <= i)
//   [Vn | O1] = [U | 0] - S_bf [W | Q]^T            (negated-A MMAs, S_bf read from TMEM)
//   O  = -gam O1 + P Vn,   o_i = scale rq_i O_i
//   S <- gam_last S + (Vn diag(d rk))^T K
//
// Roles (15 warps):
//   warp 0     TMA producer: K/Q tiles, a second copy of K for the state update, V,
//              and the gate vectors (log g, beta) of each chunk; per unit it also hands
//              the unit's record (bounds, state slot, kinds) to the chain group through
//              a small ring in shared memory and starts the unit's incoming state
//              toward L2, well before the chain group needs either;
//   warp 1     issues the chunk-local MMAs: Gram [K;Q] [K;Q]^T, then W^T and U^T;
//   warp 2     issues the serial-chain MMAs: [Vn | O1] and then O += Vn P^T, S += ...;
//   warps 3-10 chunk-local SIMT work, one chunk ahead of the chain (two threads per
//              TMEM row): the q/k norms (Gram diagonal), A and P, the triangular solve,
//              the T-derived operands, W re-layout; their first warp also scans the
//              gates of the next chunk while W and U are computed;
//   warps 11-14 chain epilogues: Vn operands, output tile, state rescale / bf16 copy,
//              initial and final states (a 16-bit pool's by TMA, in two 64-column halves
//              staged in the output stage and in the K-copy slot of the unit's last chunk,
//              whose release to the producer waits until the next unit's state is in).
// All hand-offs are mbarriers; every wait is bounded (PrefillParams::wait_ns, 200 ms by
// default) and a timeout ends the CTA's work with an error bit instead of hanging: the
// role raises a CTA-wide abort flag, every role leaves through bounded waits, and the
// drains of issued TMA loads and MMAs (always with the full bound) complete before
// TMEM is freed.
//
// Precision: every chunk product is a tcgen05 kind::f16 MMA (bf16 operands, or fp16
// when q/k/v are fp16; fp32 accumulators in TMEM) with the 128-wide head dimension on
// the M side.  K and Q enter the MMAs as the exact input tiles (the L2 norms are folded
// into fp32 diagonal factors); the two operands whose rounding reaches the state
// directly, T diag(beta) and Vn diag(d rk), are split into hi + lo halves.
//
// Masking: rows past the end of a sequence get beta = 0 and log g = 0, which makes
// their rows of T the identity and their rows of W, U and Vn exactly 0, so they
// never reach the state; their outputs are not stored.
#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <float.h>
#include <stddef.h>
#include <stdint.h>

#include "prefill.h"
#include "ptx.cuh"

namespace gdn {
// (x0, x1) *= (a0, a1) as one packed f32x2 multiply
__device__ __forceinline__ void mul2(float& x0, float& x1, float a0, float a1) {
  asm("{\n.reg .b64 t, u;\nmov.b64 t, {%0, %1};\nmov.b64 u, {%2, %3};\nmul.rn.f32x2 t, t, u;\nmov.b64 {%0, %1}, t;\n}"
      : "+f"(x0), "+f"(x1)
      : "f"(a0), "f"(a1));
}
}  // namespace gdn

namespace gdn {
namespace {

// ------------------------------------------------------------ shared memory map (bytes)
constexpr int kStagesB = 3;              // K/Q tiles (+ W, + gates) ring
constexpr uint32_t kBBytes = 32768;      // [K, then W rows dk0-63 | Q dk0-63 | K, then W rows dk64-127 | Q dk64-127]
constexpr uint32_t OFF_B = 0;
constexpr uint32_t OFF_KC = OFF_B + kStagesB * kBBytes;  // 2 x 16 KB: K for the state update (2-slot ring)
constexpr uint32_t OFF_V = OFF_KC + 2 * 16384;           // 16 KB: V [dv0-63 | dv64-127], then 16 KB:
                                                         // the output tile staged for its TMA stores
                                                         // (two 128B-swizzled halves, values 0-63 | 64-127)
constexpr uint32_t OFF_P = OFF_V + 2 * 16384;            // 2 x 8 KB:  P (64 x 64 bf16, K-major)
constexpr uint32_t OFF_WK = OFF_P + 2 * 8192;            // chunk-local work region
constexpr int kAS = 68;                  // fp32 row stride of A and T (bank-conflict free)
constexpr uint32_t WK_A = 0;             // A fp32 [64][68]            (17408 B)
constexpr uint32_t WK_X = 17408;         // solve scratch fp32 [32][32] (4096 B)
constexpr uint32_t WK_T = 24576;         // T fp32 [64][68]            (17408 B)
constexpr uint32_t WK_LW = 0;            // T diag(beta gam rk) bf16 K-major (8 KB), over A
constexpr uint32_t WK_LUHI = 8192;       // T diag(beta) hi
constexpr uint32_t WK_LULO = 16384;      // T diag(beta) lo (over A's tail and X)
constexpr uint32_t kWorkBytes = 41984;
constexpr uint32_t OFF_GATE = OFF_WK + kWorkBytes;       // 3 stages x {log g[64], beta[64]} fp32
constexpr int kVecSlots = 3;             // per-chunk vectors: written one chunk ahead of the chain
constexpr uint32_t OFF_VEC = OFF_GATE + kStagesB * 512;  // 3 slots x {gam, d*rk, rq, misc}[64] fp32
constexpr uint32_t OFF_IVEC = OFF_VEC + kVecSlots * 1024;        // chunk-local: lgscan, G, rk, beta*gam*rk, norm partials [64]
constexpr uint32_t OFF_BAR = OFF_IVEC + 2048;
constexpr int kRecSlots = 4;             // unit records the producer hands to the chain group
constexpr uint32_t OFF_REC = OFF_BAR + 512;
constexpr uint32_t kSmemUsed = OFF_REC + 512;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;        // + alignment slack

static_assert(OFF_KC % 1024 == 0 && OFF_V % 1024 == 0 && OFF_P % 1024 == 0 && OFF_WK % 1024 == 0 &&
                  (OFF_WK + WK_LUHI) % 1024 == 0 && (OFF_WK + WK_LULO) % 1024 == 0,
              "UMMA operand blocks must be 1024-byte aligned");
static_assert(WK_X + 32 * 36 * 4 <= WK_T && WK_A + 64 * kAS * 4 <= WK_X && WK_T + 64 * kAS * 4 <= kWorkBytes,
              "work region overlap");
static_assert(WK_LULO + 8192 <= WK_T, "the T-derived operands must not overwrite T");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// ------------------------------------------------------------ TMEM map (columns)
constexpr uint32_t TM_S = 0;      // S fp32 (128)
constexpr uint32_t TM_SB = 128;   // S as packed bf16 pairs (64), the A operand of the chain MMA;
                                  // between the two chain MMAs its first 32 columns hold Vd lo
constexpr uint32_t TM_VDH = 192;  // Vd hi (32 columns of packed bf16 pairs), A operand of the state update
constexpr uint32_t TM_ACC = 256;  // 2 x 128 per chunk: [U -> Vn (fp32), then Vn bf16] (64)
                                  // and [W^T -> O] (64); before the W/U products the whole
                                  // slot holds the Gram [K;Q] [K;Q]^T (128)
constexpr uint32_t kTmemCols = 512;

// ------------------------------------------------------------ roles, barriers
constexpr int kThreads = 480;
constexpr int kWarpProducer = 0, kWarpMmaLocal = 1, kWarpMmaChain = 2;
constexpr int kWgLocal = 3, kWgChain = 11;   // chunk-local group: 8 warps; chain group: 4 warps
constexpr int kLocalThreads = 256;
constexpr int kBarLocal = 1, kBarChain = 2;  // named barrier ids
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // default bound of every wait (PrefillParams::wait_ns)
constexpr int32_t kErrCu = 0x1, kErrIdx = 0x2, kErrTimeout = 0x4;

struct Bars {
  uint64_t full_b[kStagesB], full_kc[2], full_v[2];
  uint64_t empty_b[kStagesB], empty_kc[2], empty_v[2];
  uint64_t gram_done, l_ready, wu_done;
  uint64_t b_ready[2], gates_ready[2], acc_free[2];
  uint64_t c1_done, vd_ready, c2_done, s_ready;
  uint64_t drain_local, drain_chain;
  uint64_t rec_full[kRecSlots], rec_empty[kRecSlots];
  uint64_t st_full;  // the incoming state's two TMA halves have landed
  uint32_t tmem_base;
  int32_t abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

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
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// The 16-bit operand type of the tensor-core products: fp16 (F16) or bf16, as q/k/v.
template <bool F16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) { return F16 ? pack_f16(lo, hi) : pack_bf16(lo, hi); }
template <bool F16>
__device__ __forceinline__ uint16_t to16(float x) { return (uint16_t)(pack16<F16>(x, 0.f) & 0xffffu); }
// 2^x on the multi-function unit (ex2.approx.ftz: about 2 ulp, flushes subnormals).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNormEps = 1e-6f;  // x / sqrt(|x|^2 + eps) for the q/k L2 norm

// hi = bf16(x), lo = bf16(x - hi): x ~= hi + lo to ~16 significant bits.
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}
// Same split in fp16: about 22 significant bits.
__device__ __forceinline__ void split_f16(float a, float b, uint32_t& hi, uint32_t& lo) {
  __half2 h = __floats2half2_rn(a, b);
  float2 hf = __half22float2(h);
  __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}
template <bool F16>
__device__ __forceinline__ void split16(float a, float b, uint32_t& hi, uint32_t& lo) {
  if (F16) split_f16(a, b, hi, lo);
  else split_bf16(a, b, hi, lo);
}
__device__ __forceinline__ void set_error(int32_t* err, int32_t bit) { atomicOr(err, bit); }

// Read 32 consecutive floats (columns c0..c0+31) of a state row (fp32, bf16 or fp16).
__device__ __forceinline__ void load_state_chunk(const void* base, int dtype, int64_t off, int c0, float (&v)[32]) {
  if (dtype == kF32) {
    const float4* q = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + off + c0);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 x = __ldg(q + c);
      v[4 * c] = x.x; v[4 * c + 1] = x.y; v[4 * c + 2] = x.z; v[4 * c + 3] = x.w;
    }
  } else {
    const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(base) + off + c0);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 x = __ldg(q + c);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = dtype == kF16 ? __half22float2(*reinterpret_cast<const __half2*>(&w[e]))
                                       : __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
        v[8 * c + 2 * e] = f.x; v[8 * c + 2 * e + 1] = f.y;
      }
    }
  }
}
__device__ __forceinline__ void store_state_chunk(void* base, int dtype, int64_t off, int c0, const float* v32) {
  if (dtype == kF32) {
    float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + off + c0);
#pragma unroll
    for (int c = 0; c < 8; ++c) p[c] = make_float4(v32[4 * c], v32[4 * c + 1], v32[4 * c + 2], v32[4 * c + 3]);
  } else if (dtype == kF16) {
    uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(base) + off + c0);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      p[c] = make_uint4(pack_f16(v32[8 * c], v32[8 * c + 1]), pack_f16(v32[8 * c + 2], v32[8 * c + 3]),
                        pack_f16(v32[8 * c + 4], v32[8 * c + 5]), pack_f16(v32[8 * c + 6], v32[8 * c + 7]));
  } else {
    uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + off + c0);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      p[c] = make_uint4(pack_bf16(v32[8 * c], v32[8 * c + 1]), pack_bf16(v32[8 * c + 2], v32[8 * c + 3]),
                        pack_bf16(v32[8 * c + 4], v32[8 * c + 5]), pack_bf16(v32[8 * c + 6], v32[8 * c + 7]));
  }
}


// ------------------------------------------------------------ per-unit bookkeeping
struct Unit {
  int64_t bos, eos;   // token rows of this unit (a whole sequence or one segment of it)
  int64_t slot;       // state slot of the sequence in the caller's pools
  int64_t in_ws, out_ws;  // workspace blocks (split-K)
  int n, h, hq, hv, nch;
  int c_off;              // chunks of the sequence before this unit's first one (split-K)
  int in_kind, out_kind;  // see kIn* / kOut*
  bool zero_v, write_out;
  bool idle;          // an index of the unit order that holds no unit (split-K plans)
  int32_t err;        // device error bits this unit raises (reported by the chain warpgroup)
};
constexpr int kInPool = 0, kInZero = 1, kInIdentity = 2, kInWs = 3;
constexpr int kOutPool = 0, kOutWs = 1, kOutNone = 2;

// The u-th unit of this launch.  Mode 0: (sequence, head).  Mode 1: per (sequence, head)
// 2P-3 kinds: segment 0 (outputs written, final state -> S_1), then M_p (from the identity,
// v = 0) and N_p (from zero) of segments p = 1..P-2.  Mode 2: per (sequence, head) the
// segments p = 1..P-1 from S_p; the last one writes the caller's final state.  A split
// plan may order the units in runs (PrefillParams::runs).
// Not inlined: it runs once per unit per role, and one shared copy keeps the hot
// per-chunk code of every role small enough for the instruction caches.
__device__ __noinline__ Unit unit_info(const PrefillParams& p, int64_t u) {
  Unit U{};
  int n, kind = 0;
  const int P = p.splits;
  const int K = p.mode == 1 ? 2 * P - 3 : (p.mode == 2 ? P - 1 : 1);
  if (p.mode != 0) {
    int32_t nh, k;
    if (!split_unit(p, u, &nh, &k)) {
      U.idle = true;
      return U;
    }
    kind = k;
    n = nh / p.H;
    U.h = nh - n * p.H;
  } else if (p.n_units <= 0x7fffffff) {  // 32-bit divisions: the 64-bit ones are emulated and slow
    const uint32_t u32 = (uint32_t)u, nh = u32 / (uint32_t)K;
    kind = (int)(u32 - nh * (uint32_t)K);
    n = (int)(nh / (uint32_t)p.H);
    U.h = (int)(nh - (uint32_t)n * (uint32_t)p.H);
  } else {
    const int64_t nh = u / K;
    kind = (int)(u - nh * K);
    n = (int)(nh / p.H);
    U.h = (int)(nh - (int64_t)n * p.H);
  }
  U.n = n;
  U.c_off = 0;
  U.hq = U.h / (p.H / p.H_qk);
  U.hv = U.h / (p.H / p.H_v);
  const int64_t bos = load_index(p.cu, p.cu_dtype, n);
  const int64_t eos = load_index(p.cu, p.cu_dtype, n + 1);
  U.slot = p.state_idx ? load_index(p.state_idx, p.idx_dtype, n) : (int64_t)n;
  U.err = 0;
  if (bos < 0 || eos < bos || eos > p.T) U.err = kErrCu;
  else if ((p.s_in && (U.slot < 0 || U.slot >= p.sin_slots)) ||
           (p.s_out && (U.slot < 0 || U.slot >= p.sout_slots)))
    U.err = kErrIdx;
  U.bos = bos;
  U.eos = eos;
  U.in_kind = kInPool;
  U.out_kind = kOutPool;
  U.in_ws = U.out_ws = 0;
  U.zero_v = false;
  U.write_out = true;
  if (p.mode != 0 && !U.err) {
    const int64_t base = ((int64_t)n * p.H + U.h) * split_ws_blocks(P);
    const int64_t nch_all = (eos - bos + kChunk - 1) / kChunk;
    int seg;
    if (p.mode == 1) {
      if (kind == 0) { seg = 0; U.out_kind = kOutWs; U.out_ws = base; }
      else if (kind <= P - 2) { seg = kind; U.in_kind = kInIdentity; U.zero_v = true; U.write_out = false;
                                U.out_kind = kOutWs; U.out_ws = base + (P - 1) + (seg - 1); }
      else { seg = kind - (P - 2); U.in_kind = kInZero; U.write_out = false;
             U.out_kind = kOutWs; U.out_ws = base + (P - 1) + (P - 2) + (seg - 1); }
    } else {
      seg = kind + 1;
      U.in_kind = kInWs;
      U.in_ws = base + (seg - 1);
      U.out_kind = (seg == P - 1) ? kOutPool : kOutNone;
    }
    const int64_t c0 = nch_all * p.seg_num[seg] / p.seg_den, c1 = nch_all * p.seg_num[seg + 1] / p.seg_den;
    U.bos = bos + c0 * kChunk;
    U.eos = (bos + c1 * kChunk < eos) ? bos + c1 * kChunk : eos;
    U.c_off = (int)c0;
  }
  U.nch = U.err ? 0 : (int)((U.eos - U.bos + kChunk - 1) / kChunk);
  return U;
}

// Number of chunks this CTA walks (over its units u = blockIdx.x + k * gridDim.x).
__device__ __noinline__ int cta_items(const PrefillParams& p) {
  int n = 0;
  if (p.mode == 0 && p.n_units <= 0x7fffffff) {
    // one unit per (sequence, head): the same count as the sum of unit_info(p, u).nch
    // (units with a bad bound or state index hold no chunks), with the index loads of
    // several units in flight at once
    const uint32_t H = (uint32_t)p.H, nu = (uint32_t)p.n_units;
#pragma unroll 4
    for (uint32_t u = blockIdx.x; u < nu; u += gridDim.x) {
      const uint32_t s = u / H;
      const int64_t bos = load_index(p.cu, p.cu_dtype, s), eos = load_index(p.cu, p.cu_dtype, s + 1);
      const int64_t slot = p.state_idx ? load_index(p.state_idx, p.idx_dtype, s) : (int64_t)s;
      const bool bad = bos < 0 || eos < bos || eos > p.T || (p.s_in && (slot < 0 || slot >= p.sin_slots)) ||
                       (p.s_out && (slot < 0 || slot >= p.sout_slots));
      n += bad ? 0 : (int)((eos - bos + kChunk - 1) / kChunk);
    }
    return n;
  }
  for (int64_t u = blockIdx.x; u < p.n_units; u += gridDim.x) n += unit_info(p, u).nch;
  return n;
}

struct Smem {
  uint8_t* base;
  Bars* bars;
  __device__ uint8_t* B(int s3) const { return base + OFF_B + s3 * kBBytes; }
  __device__ uint8_t* KC(int s) const { return base + OFF_KC + s * 16384; }
  __device__ uint8_t* V() const { return base + OFF_V; }
  __device__ uint8_t* stage() const { return base + OFF_V + 16384; }
  __device__ uint8_t* P(int s) const { return base + OFF_P + s * 8192; }
  __device__ uint8_t* wk() const { return base + OFF_WK; }
  __device__ float* gate_lg(int s3) const { return reinterpret_cast<float*>(base + OFF_GATE + s3 * 512); }
  __device__ float* gate_beta(int s3) const { return gate_lg(s3) + 64; }
  // per-chunk vectors handed from the chunk-local warpgroup to the chain warpgroup
  __device__ float* vgam(int s) const { return reinterpret_cast<float*>(base + OFF_VEC + s * 1024); }
  __device__ float* vdk(int s) const { return vgam(s) + 64; }    // e^{G_last - G_j} rk_j
  __device__ float* vrq(int s) const { return vgam(s) + 128; }   // scale * rq_i
  __device__ float* vmisc(int s) const { return vgam(s) + 192; } // [0] = gam_last
  __device__ float* ivec(int k) const { return reinterpret_cast<float*>(base + OFF_IVEC) + 64 * k; }
  __device__ Unit* rec(int slot) const { return reinterpret_cast<Unit*>(base + OFF_REC) + slot; }
};
static_assert(kRecSlots * sizeof(Unit) <= 512 && OFF_REC % alignof(Unit) == 0, "unit records");

__device__ __forceinline__ bool aborted(const Bars* b) {
  return *reinterpret_cast<const volatile int32_t*>(&b->abort_flag) != 0;
}
__device__ __forceinline__ void raise_abort(const PrefillParams& p, Bars* b) {
  *reinterpret_cast<volatile int32_t*>(&b->abort_flag) = 1;
  set_error(p.dev_err, kErrTimeout);
}

// ------------------------------------------------------------ warp 0: loads
__device__ __forceinline__ void run_producer(const PrefillParams& p, const Smem S, int lane) {
  Bars* bars = S.bars;
  // loads issued per ring slot (kept in registers: indexed only through selects)
  uint32_t issued_b0 = 0, issued_b1 = 0, issued_b2 = 0, issued_v0 = 0, issued_v1 = 0, issued_kc0 = 0, issued_kc1 = 0;
  int i = 0;
  bool ok = true;
  int jr = 0;  // units of this CTA so far
  for (int64_t u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++jr) {
    const Unit U = unit_info(p, u);
    {  // hand the unit's record to the chain group, and start its incoming state toward L2
      const int rs = jr % kRecSlots;
      bool w = jr < kRecSlots || mbar_wait(&bars->rec_empty[rs], ((jr / kRecSlots) - 1) & 1, p.wait_ns);
      ok = __all_sync(0xffffffffu, w && !aborted(bars));
      if (!ok) break;
      if (lane == 0) {
        *S.rec(rs) = U;
        mbar_arrive(&bars->rec_full[rs]);  // releases the record
        if (!U.idle && !U.err && U.nch > 0) {
          if (U.in_kind == kInPool && p.s_in) {
            const int es = p.sin_dtype == kF32 ? 4 : 2;
            const char* src = reinterpret_cast<const char*>(p.s_in) + (U.slot * p.sin_slot + (int64_t)U.h * p.sin_head) * es;
            if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) bulk_prefetch_l2(src, (uint32_t)(kHeadDim * kHeadDim * es));
          } else if (U.in_kind == kInWs) {
            bulk_prefetch_l2(p.ws + U.in_ws * (kHeadDim * kHeadDim), (uint32_t)(kHeadDim * kHeadDim * 4));
          }
        }
      }
    }
    for (int c = 0; c < U.nch; ++c, ++i) {
      const int s3 = i % kStagesB, s = i & 1;
      const int64_t t0 = U.bos + (int64_t)c * kChunk;
      const int nvalid = (U.eos - t0 < kChunk) ? (int)(U.eos - t0) : kChunk;
      // every wait is made by the whole warp (see run_mma_local), lane 0 issues the copies
      bool w = true;
      if (i >= kStagesB) w = mbar_wait(&bars->empty_b[s3], ((i / kStagesB) - 1) & 1, p.wait_ns);
      ok = __all_sync(0xffffffffu, w && !aborted(bars));
      if (!ok) break;
      // gate vectors of the chunk: log g (clamped to [log FLT_MIN, 0]) and beta; 0 past the
      // sequence end
      float* gl = S.gate_lg(s3);
      float* gb = S.gate_beta(s3);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int r = lane + 32 * k;
        float lg = 0.f, bt = 0.f;
        if (r < nvalid) {
          const int64_t t = t0 + r;
          if (p.g) lg = fminf(__logf(fmaxf(load_real(p.g, p.g_dtype, t * p.g_st + (int64_t)U.h * p.g_sh), FLT_MIN)), 0.f);
          bt = p.beta ? load_real(p.beta, p.b_dtype, t * p.b_st + (int64_t)U.h * p.b_sh) : 1.f;
        }
        gl[r] = lg;
        gb[r] = bt;
      }
      __syncwarp();
      if (lane == 0) {
        uint8_t* B = S.B(s3);
        mbar_arrive_expect_tx(&bars->full_b[s3], kBBytes);  // also publishes the gate stores
        tma_load_3d(B + 0, &p.tm_k, &bars->full_b[s3], 0, U.hq, (int)t0);
        tma_load_3d(B + 8192, &p.tm_q, &bars->full_b[s3], 0, U.hq, (int)t0);
        tma_load_3d(B + 16384, &p.tm_k, &bars->full_b[s3], 64, U.hq, (int)t0);
        tma_load_3d(B + 24576, &p.tm_q, &bars->full_b[s3], 64, U.hq, (int)t0);
        issued_b0 += (s3 == 0); issued_b1 += (s3 == 1); issued_b2 += (s3 == 2);
      }
      // one V slot: item i's tile goes in once the U^T product of item i - 1 has read it
      if (i >= 1) w = mbar_wait(&bars->empty_v[0], (i - 1) & 1, p.wait_ns);
      w = __all_sync(0xffffffffu, w);
      if (w && lane == 0) {
        mbar_arrive_expect_tx(&bars->full_v[0], 16384);
        tma_load_3d(S.V(), &p.tm_v, &bars->full_v[0], 0, U.hv, (int)t0);
        tma_load_3d(S.V() + 8192, &p.tm_v, &bars->full_v[0], 64, U.hv, (int)t0);
        ++issued_v0;
      }
      if (w && i >= 2) w = mbar_wait(&bars->empty_kc[s], ((i >> 1) - 1) & 1, p.wait_ns);
      w = __all_sync(0xffffffffu, w);
      if (w && lane == 0) {
        mbar_arrive_expect_tx(&bars->full_kc[s], 16384);
        tma_load_3d(S.KC(s), &p.tm_k, &bars->full_kc[s], 0, U.hq, (int)t0);
        tma_load_3d(S.KC(s) + 8192, &p.tm_k, &bars->full_kc[s], 64, U.hq, (int)t0);
        issued_kc0 += (s == 0); issued_kc1 += (s == 1);
      }
      ok = w;
      if (!ok) break;
    }
  }
  if (!ok && lane == 0) {
    raise_abort(p, bars);
    // let issued tile loads land before the CTA's shared memory goes away
    const uint32_t nb[3] = {issued_b0, issued_b1, issued_b2};
    for (int b = 0; b < kStagesB; ++b)
      if (nb[b]) mbar_wait(&bars->full_b[b], (nb[b] - 1) & 1, kWaitLimitNs);
    const uint32_t nv[2] = {issued_v0, issued_v1}, nk[2] = {issued_kc0, issued_kc1};
    for (int b = 0; b < 2; ++b) {
      if (nv[b]) mbar_wait(&bars->full_v[b], (nv[b] - 1) & 1, kWaitLimitNs);
      if (nk[b]) mbar_wait(&bars->full_kc[b], (nk[b] - 1) & 1, kWaitLimitNs);
    }
  }
}

// ------------------------------------------------------------ warp 1: chunk-local MMAs
// The whole warp runs the loop and waits (a lone waiting lane in an otherwise parked warp
// was measured to wake 0.6-0.8 us after its barrier completed); lane 0 issues.
template <bool F16>
__device__ __forceinline__ void run_mma_local(const PrefillParams& p, const Smem S, uint32_t tmem, bool leader) {
  Bars* bars = S.bars;
  const uint32_t id_gram = idesc_16_f32(F16, 128, 128, 0, 0, 0);
  const uint32_t id_wu = idesc_16_f32(F16, 128, 64, 1, 0, 0);
  const uint32_t lw = smem_u32(S.wk() + WK_LW), luh = smem_u32(S.wk() + WK_LUHI), lul = smem_u32(S.wk() + WK_LULO);
  const int n_items = cta_items(p);
  bool ok = true;
  // Descriptor bases; a step adds its byte offset / 16 to the start-address field (shared
  // addresses stay below 2^18, so the 14-bit field never carries).
  const uint64_t d_lw = sdesc_sw128(lw, 16, 1024), d_luh = sdesc_sw128(luh, 16, 1024),
                 d_lul = sdesc_sw128(lul, 16, 1024);
  // Step k issues W^T and U^T of chunk k - 1, then the Gram of chunk k.
  for (int k = 0; k <= n_items && ok; ++k) {
    if (k >= 1) {
      const int i = k - 1, s3 = i % kStagesB, s = i & 1;
      ok = mbar_wait(&bars->l_ready, i & 1, p.wait_ns) && mbar_wait(&bars->full_v[0], i & 1, p.wait_ns);
      ok = __all_sync(0xffffffffu, ok);  // one decision for the warp
      if (!ok) break;
      tc_fence_after();
      const uint64_t d_k = sdesc_sw128(smem_u32(S.B(s3)), 16384, 1024), d_v = sdesc_sw128(smem_u32(S.V()), 8192, 1024);
      const uint32_t acc = tmem + TM_ACC + s * 128;
      // W^T = K^T (T diag(beta gam rk))^T into the O half (A = K as MN-major: dk blocks 16 KB
      // apart); U^T = V^T (T diag(beta))^T into the U half, hi then lo halves of T diag(beta)
      if (leader) {
#pragma unroll
        for (int st = 0; st < 4; ++st) mma_ss(acc + 64, d_k + st * 128, d_lw + st * 2, id_wu, st > 0);
#pragma unroll
        for (int st = 0; st < 4; ++st) mma_ss(acc, d_v + st * 128, d_luh + st * 2, id_wu, st > 0);
#pragma unroll
        for (int st = 0; st < 4; ++st) mma_ss(acc, d_v + st * 128, d_lul + st * 2, id_wu, 1);
        mma_commit(&bars->wu_done);
        mma_commit(&bars->empty_v[0]);
      }
      __syncwarp();
    }
    if (k < n_items) {
      // Gram [K;Q] [K;Q]^T of chunk k into its whole accumulator slot: M = N = 128 (k rows,
      // then q rows), K = 128 (two 64-wide atoms); its diagonal holds the q/k norms
      const int s3 = k % kStagesB, s = k & 1;
      bool w = mbar_wait(&bars->full_b[s3], (k / kStagesB) & 1, p.wait_ns);
      if (w && k >= 2) w = mbar_wait(&bars->acc_free[s], ((k >> 1) - 1) & 1, p.wait_ns);
      if (!__all_sync(0xffffffffu, w && !aborted(bars))) { ok = false; break; }
      tc_fence_after();
      const uint64_t d_b = sdesc_sw128(smem_u32(S.B(s3)), 16, 1024);
      const uint32_t dst = tmem + TM_ACC + s * 128;
      if (leader) {
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          const uint64_t d = d_b + ((st >> 2) * 16384 + (st & 3) * 32) / 16;
          mma_ss(dst, d, d, id_gram, st > 0);
        }
        mma_commit(&bars->gram_done);
      }
      __syncwarp();
    }
  }
  if (!ok && leader) raise_abort(p, bars);
  if (leader) mma_commit(&bars->drain_local);  // everything issued has completed once this arrives
  __syncwarp();
  mbar_wait(&bars->drain_local, 0, kWaitLimitNs);  // drains keep the full bound
}

// ------------------------------------------------------------ warp 2: serial-chain MMAs
template <bool F16>
__device__ __forceinline__ void run_mma_chain(const PrefillParams& p, const Smem S, uint32_t tmem, bool leader) {
  Bars* bars = S.bars;
  const uint32_t id_c1w = idesc_16_f32(F16, 128, 64, 0, 1, 1);  // Vn = U - S W^T (W: MN-major rows dk)
  const uint32_t id_c1q = idesc_16_f32(F16, 128, 64, 0, 0, 1);  // O1' = -S Q^T  (Q: K-major rows i)
  const uint32_t id_o2 = idesc_16_f32(F16, 128, 64, 0, 0, 0);   // O += Vn P^T
  const uint32_t id_s = idesc_16_f32(F16, 128, 128, 0, 1, 0);   // S += Vd^T K
  const int n_items = cta_items(p);
  bool ok = true;
  for (int i = 0; i < n_items && ok; ++i) {
    {
      const int s3 = i % kStagesB, s = i & 1;
      const uint32_t acc = tmem + TM_ACC + s * 128;
      ok = mbar_wait(&bars->b_ready[s], (i >> 1) & 1, p.wait_ns) && mbar_wait(&bars->s_ready, i & 1, p.wait_ns);
      ok = __all_sync(0xffffffffu, ok && !aborted(bars));  // one decision for the warp
      if (!ok) break;
      tc_fence_after();
      const uint32_t b_a = smem_u32(S.B(s3));
      const uint64_t d_w = sdesc_sw128(b_a, 8192, 1024), d_q = sdesc_sw128(b_a + 8192, 16, 1024);
      if (leader) {
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          mma_ts(acc, tmem + TM_SB + st * 8, d_w + ((st >> 2) * 16384 + (st & 3) * 2048) / 16, id_c1w, 1);
          mma_ts(acc + 64, tmem + TM_SB + st * 8, d_q + ((st >> 2) * 16384 + (st & 3) * 32) / 16, id_c1q, st > 0);
        }
        mma_commit(&bars->c1_done);
        mma_commit(&bars->empty_b[s3]);
      }
      __syncwarp();
      ok = mbar_wait(&bars->vd_ready, i & 1, p.wait_ns) && mbar_wait(&bars->full_kc[s], (i >> 1) & 1, p.wait_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint64_t d_p = sdesc_sw128(smem_u32(S.P(s)), 16, 1024), d_kc = sdesc_sw128(smem_u32(S.KC(s)), 8192, 1024);
      if (leader) {
#pragma unroll
        for (int st = 0; st < 4; ++st) mma_ts(acc + 64, acc + st * 8, d_p + st * 2, id_o2, 1);
#pragma unroll
        for (int st = 0; st < 4; ++st) mma_ts(tmem + TM_S, tmem + TM_VDH + st * 8, d_kc + st * 128, id_s, 1);
#pragma unroll
        for (int st = 0; st < 4; ++st) mma_ts(tmem + TM_S, tmem + TM_SB + st * 8, d_kc + st * 128, id_s, 1);
        mma_commit(&bars->c2_done);
      }
      __syncwarp();
    }
  }
  if (!ok && leader) raise_abort(p, bars);
  if (leader) mma_commit(&bars->drain_chain);
  __syncwarp();
  mbar_wait(&bars->drain_chain, 0, kWaitLimitNs);  // drains keep the full bound
}

// ------------------------------------------------------------ T = (I + A)^-1
constexpr int kXS = 36;  // fp32 row stride of the 32 x 32 merge product X (bank-conflict free B reads)

// d = sum_{k < 32} A[m][k] B[k][n] for the 16 x 8 tile (m < 16, n < 8) at A, B (fp32
// row-major in shared memory, row strides lda, ldb), on m16n8k16 bf16 products with
// each operand split into bf16 hi + lo: hi*hi + (lo*hi + hi*lo), about 16 significant
// bits per operand (the lo*lo term, ~2^-18 relative, is dropped).  Warp-collective.
__device__ __forceinline__ void tile16x8_bf16x3(const float* A, int lda, const float* B, int ldb, int lane,
                                                float (&d)[4]) {
  const int g = lane >> 2, t = lane & 3;
  float d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] = 0.f;
#pragma unroll
  for (int s = 0; s < 2; ++s) {  // per 16-wide k step: fragments, then the hi*hi and cross-term chains
    const int k0 = 16 * s;
    uint32_t ah[4], al[4], bh[2], bl[2];
    const float2 a0 = *reinterpret_cast<const float2*>(A + g * lda + k0 + 2 * t);
    const float2 a1 = *reinterpret_cast<const float2*>(A + (g + 8) * lda + k0 + 2 * t);
    const float2 a2 = *reinterpret_cast<const float2*>(A + g * lda + k0 + 2 * t + 8);
    const float2 a3 = *reinterpret_cast<const float2*>(A + (g + 8) * lda + k0 + 2 * t + 8);
    split_bf16(a0.x, a0.y, ah[0], al[0]);
    split_bf16(a1.x, a1.y, ah[1], al[1]);
    split_bf16(a2.x, a2.y, ah[2], al[2]);
    split_bf16(a3.x, a3.y, ah[3], al[3]);
    split_bf16(B[(k0 + 2 * t) * ldb + g], B[(k0 + 2 * t + 1) * ldb + g], bh[0], bl[0]);
    split_bf16(B[(k0 + 2 * t + 8) * ldb + g], B[(k0 + 2 * t + 9) * ldb + g], bh[1], bl[1]);
    mma_sync_bf16(d1, al, bh);
    mma_sync_bf16(d, ah, bh);
    mma_sync_bf16(d1, ah, bl);
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] += d1[e];
}
// A: strictly lower fp32 [64][kAS] (only entries below the diagonal are read).  Writes
// the lower triangle of T (diagonal included) into sT; the blocks above the 16 x 16
// diagonal blocks are zero already (cleared once per CTA, never written).  Blocked: the
// four 16 x 16 diagonal blocks by forward substitution (one column per thread, no
// barrier inside), then T21 = -T22 (A21 T11) for 16 -> 32 and 32 -> 64.
// kLocalThreads threads (at = 0..255) synchronised on named barrier `bar`.
__device__ __forceinline__ void solve_unit_lower(const float* sA, float* sT, float* sX, int at, int bar) {
  constexpr int NT = kLocalThreads;
  if (at < 64) {  // four 16 x 16 diagonal blocks, one column per thread, by forward substitution
    const int base = (at >> 4) * 16, m = at & 15;
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float* ar = sA + (base + i) * kAS + base;
      float acc = (i == m) ? 1.f : 0.f;
#pragma unroll
      for (int j = 0; j < i; ++j) acc = fmaf(-ar[j], t[j], acc);
      t[i] = acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sT[(base + i) * kAS + base + m] = t[i];
  }
  named_sync(bar, NT);
  {  // 16 -> 32, X = A21 T11 (two elements per thread)
    const int pb = at >> 7, q = at & 127, c = q & 15, r0 = (q >> 4) * 2, base = 32 * pb;
    float x[2] = {0.f, 0.f};
#pragma unroll
    for (int k4 = 0; k4 < 16; k4 += 4) {
      float tk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) tk[e] = sT[(base + k4 + e) * kAS + base + c];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const float4 a = *reinterpret_cast<const float4*>(sA + (base + 16 + r0 + rr) * kAS + base + k4);
        x[rr] = fmaf(a.x, tk[0], fmaf(a.y, tk[1], fmaf(a.z, tk[2], fmaf(a.w, tk[3], x[rr]))));
      }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) sX[pb * 256 + (r0 + rr) * 16 + c] = x[rr];
  }
  named_sync(bar, NT);
  {  // T21 = -T22 X
    const int pb = at >> 7, q = at & 127, c = q & 15, r0 = (q >> 4) * 2, base = 32 * pb;
    float y[2] = {0.f, 0.f};
#pragma unroll
    for (int k4 = 0; k4 < 16; k4 += 4) {
      float xk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) xk[e] = sX[pb * 256 + (k4 + e) * 16 + c];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const float4 a = *reinterpret_cast<const float4*>(sT + (base + 16 + r0 + rr) * kAS + base + 16 + k4);
        y[rr] = fmaf(a.x, xk[0], fmaf(a.y, xk[1], fmaf(a.z, xk[2], fmaf(a.w, xk[3], y[rr]))));
      }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) sT[(base + 16 + r0 + rr) * kAS + base + c] = -y[rr];
  }
  named_sync(bar, NT);
  // 32 -> 64 on the warp-level tensor path, one 16 x 8 output tile per warp: step 0 forms
  // X = A21 T11, step 1 writes T21 = -T22 X
  const int w = at >> 5, lane = at & 31, m0 = (w >> 2) * 16, n0 = (w & 3) * 8, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int step = 0; step < 2; ++step) {
    const float* a = step == 0 ? sA + (32 + m0) * kAS : sT + (32 + m0) * kAS + 32;
    const float* b = step == 0 ? sT + n0 : sX + n0;
    float* d_out = step == 0 ? sX + m0 * kXS + n0 : sT + (32 + m0) * kAS + n0;
    const int ldd = step == 0 ? kXS : kAS;
    const float sign = step == 0 ? 1.f : -1.f;
    float d[4];
    tile16x8_bf16x3(a, kAS, b, step == 0 ? kAS : kXS, lane, d);
    *reinterpret_cast<float2*>(d_out + g * ldd + 2 * t) = make_float2(sign * d[0], sign * d[1]);
    *reinterpret_cast<float2*>(d_out + (g + 8) * ldd + 2 * t) = make_float2(sign * d[2], sign * d[3]);
    named_sync(bar, NT);
  }
}

// ------------------------------------------------------------ warps 3-10: chunk-local SIMT work
// Two threads own each TMEM row r (hf = 0, 1) and split its columns.
// Columns j0..j0+15 of one decay-weighted Gram row: v_j = f rk_j 2^{G2_i - G2_j} gram_j
// (G2 = G log2 e) for j < lim, else 0, with the key factor folded into the exponent:
// rk_j 2^{G2_i - G2_j} = 2^{G2_i - H_j}, H_j = G2_j - log2 rk_j.  Branch-free: every lane
// evaluates, and a select (not a product, as the exponent may overflow to inf above the
// diagonal) keeps j < lim; a per-lane branch here would diverge per element.
__device__ __forceinline__ void decay_row16(const uint32_t* g, const float* sH, int j0,
                                            float G2i, float f, int lim, float (&v)[16]) {
#pragma unroll
  for (int j4 = 0; j4 < 16; j4 += 4) {
    const float4 hj = *reinterpret_cast<const float4*>(sH + j0 + j4);
    const float hh[4] = {hj.x, hj.y, hj.z, hj.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = (f * __uint_as_float(g[j4 + e])) * fast_exp2(G2i - hh[e]);
      v[j4 + e] = (j0 + j4 + e < lim) ? x : 0.f;
    }
  }
}

// Gates of chunk j (step 1 of the chunk-local work), on one warp: the in-chunk cumulative
// log-gate G (log2 units), gam = 2^G and gam_last, all the chain needs before the chunk's
// Gram (and with it the q/k norms) exists.  Runs one chunk ahead, while the W/U products
// of the previous chunk are on the tensor pipe; the other warps of the group skip it.
// Returns false on a timeout or abort (the caller folds that into its next group barrier).
__device__ __forceinline__ bool local_gates_warp(const Smem S, int j, int lane, uint64_t wait_ns) {
  Bars* bars = S.bars;
  const int s3 = j % kStagesB, sv = j % kVecSlots;
  const bool w = mbar_wait(&bars->full_b[s3], (j / kStagesB) & 1, wait_ns) && !aborted(bars);
  if (!__all_sync(0xffffffffu, w)) return false;  // one decision for the warp (it shuffles below)
  const float2 x = *reinterpret_cast<const float2*>(S.gate_lg(s3) + 2 * lane);  // rows 2l, 2l+1
  float incl = x.x + x.y;  // inclusive scan of the row-pair sums
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.f;
  const float G0 = excl + x.x, G1 = G0 + x.y;  // log g <= 0: G never increases
  const float g0 = G0 * kLog2e, g1 = G1 * kLog2e, e0 = fast_exp2(g0), e1 = fast_exp2(g1);
  *reinterpret_cast<float2*>(S.ivec(1) + 2 * lane) = make_float2(g0, g1);
  *reinterpret_cast<float2*>(S.vgam(sv) + 2 * lane) = make_float2(e0, e1);
  if (lane == 31) S.vmisc(sv)[0] = e1;
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars->gates_ready[j & 1]);
  return true;
}

template <bool F16>
__device__ __forceinline__ void run_local_wg(const PrefillParams& p, const Smem S, uint32_t tmem, int warp, int lane) {
  Bars* bars = S.bars;
  constexpr int NT = kLocalThreads;
  const int at = threadIdx.x - 32 * kWgLocal;  // 0..255
  const int hf = (warp - kWgLocal) >> 2;       // column half of the row this thread works on
  const int r = 32 * (warp & 3) + lane;        // TMEM lane / row
  const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  float* sA = reinterpret_cast<float*>(S.wk() + WK_A);
  float* sT = reinterpret_cast<float*>(S.wk() + WK_T);
  float* sX = reinterpret_cast<float*>(S.wk() + WK_X);
  const float* sG = S.ivec(1);  // in-chunk cumulative log g (log2 units), written by the gate warp
  float* sRk = S.ivec(2);       // key norm factors rk
  float* sF1 = S.ivec(3);       // beta gam rk
  float* sH = S.ivec(4);        // G_j - log2 rk_j: the key factor folded into the exponent
  const int n_items = cta_items(p);
  // T is lower triangular: its blocks above the 16 x 16 diagonal blocks (the upper-right
  // 16 x 16 of each 32 x 32 diagonal block, and the upper-right 32 x 32) are zero for
  // every chunk and nothing else writes them, so they are cleared once here.
  for (int e = at; e < 1536; e += NT) {
    int rr, cc;
    if (e < 1024) { rr = e >> 5; cc = 32 + (e & 31); }
    else { const int f = e - 1024, blk = f >> 8; rr = 32 * blk + ((f >> 4) & 15); cc = 32 * blk + 16 + (f & 15); }
    sT[rr * kAS + cc] = 0.f;
  }
  // Rotated loop: step k runs the gates of item k, the tail (W^T read-out) of item k - 1
  // -- which overlaps the W/U products -- and the head (A, P, solve, operands) of item k,
  // so each piece of code appears once.
  int64_t u = blockIdx.x;
  Unit U;
  U.nch = 0;
  int c = 0;
  bool ok = true;
  for (int k = 0; k <= n_items && ok; ++k) {
    const bool gok = k >= n_items || at >= 32 || local_gates_warp(S, k, lane, p.wait_ns);
    if (k >= 1) {
      const int i = k - 1, s3 = i % kStagesB, s = i & 1;
      const uint32_t go = trow + TM_ACC + s * 128 + 64;
      bool w;
      // (6) W^T (TMEM, row dk) -> rows dk of the MN-major B operand in the K slots of B (the
      //     chain MMA then overwrites these columns with -S Q^T)
      w = mbar_wait(&bars->wu_done, i & 1, p.wait_ns);
      ok = named_sync_and(kBarLocal, NT, w && gok);
      if (!ok) break;
      tc_fence_after();
      {
        uint8_t* wslot = S.B(s3) + (r >> 6) * 16384;
        const int wr = r & 63;
        uint32_t rr[32];
        tmem_ld32(go + 32 * hf, rr);
        tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            pk[e] = pack16<F16>(__uint_as_float(rr[8 * q4 + 2 * e]), __uint_as_float(rr[8 * q4 + 2 * e + 1]));
          *reinterpret_cast<uint4*>(wslot + sw128_chunk(wr, 4 * hf + q4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(kBarLocal, NT);
      if (at == 0) mbar_arrive(&bars->b_ready[s]);
    }
    if (k < n_items) {
      while (c >= U.nch && u < p.n_units) {  // the unit of item k (units without chunks hold no item)
        U = unit_info(p, u);
        u += gridDim.x;
        c = 0;
      }
      ++c;
      const int i = k, s3 = i % kStagesB, s = i & 1;
      const float* gbeta = S.gate_beta(s3);
      bool w;
      // (3) the q/k norms from the Gram diagonal, then Gram rows 16 columns at a time, this
      //     thread's half: k rows -> A (fp32), q rows -> P (bf16)
      w = mbar_wait(&bars->gram_done, i & 1, p.wait_ns);
      ok = named_sync_and(kBarLocal, NT, w && gok);
      if (!ok) break;
      tc_fence_after();
      // [K;Q][K;Q]^T: columns 0-63 against the keys, 64-127 against the queries
      const uint32_t ga = trow + TM_ACC + s * 128;
      const bool is_a = r < 64;
      const int ri = r & 63;
      {
        // Row r's own norm |x_r|^2 is the diagonal entry, which lies in the 32 columns this
        // thread reads when hf is the half of its row (register lane, as r & 31 = lane).
        const int sv = i % kVecSlots;
        if (hf == (ri >> 5)) {
          float rn = 1.f, lrn = 0.f;
          if (p.l2norm) {
            float d = 0.f;
#pragma unroll 1
            for (int q16 = 0; q16 < 32; q16 += 16) {
              uint32_t g[16];
              tmem_ld16(ga + (is_a ? 0 : 64) + 32 * hf + q16, g);
              tmem_ld_wait();
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) d = (q16 + jj == lane) ? __uint_as_float(g[jj]) : d;
            }
            rn = rsqrtf(d + kNormEps);
            lrn = 0.5f * __log2f(d + kNormEps);
          }
          if (is_a) {
            sRk[ri] = rn;
            sH[ri] = sG[ri] + lrn;
            sF1[ri] = gbeta[ri] * S.vgam(sv)[ri] * rn;
            S.vdk(sv)[ri] = fast_exp2(sG[63] - sG[ri]) * rn;
          } else {
            S.vrq(sv)[ri] = p.scale * rn;
          }
        }
        named_sync(kBarLocal, NT);
      }
      {
        // This thread's 32 columns j0..j0+31 of Gram row r (k rows -> A, q rows -> P), 16 at a
        // time.  Blocks entirely right of the warp's 32 rows are skipped (A: never read) or
        // zero (P).
        const int j0 = 32 * hf, wr = 32 * ((warp & 3) & 1);  // first row of the warp within its matrix
        const bool live = j0 <= wr;
        const float f = is_a ? gbeta[ri] * sRk[ri] : 1.f, G2i = sG[ri];
        const int lim = is_a ? ri : ri + 1;
        uint8_t* sP = S.P(s);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          const int jh = j0 + 16 * h;
          float v[16];
          if (live) {
            uint32_t g[16];
            tmem_ld16(ga + jh, g);
            tmem_ld_wait();
            decay_row16(g, sH, jh, G2i, f, lim, v);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = 0.f;
          }
          if (is_a) {
            if (live) {
              float* arow = sA + ri * kAS + jh;
#pragma unroll
              for (int j4 = 0; j4 < 16; j4 += 4)
                *reinterpret_cast<float4*>(arow + j4) = make_float4(v[j4], v[j4 + 1], v[j4 + 2], v[j4 + 3]);
            }
          } else {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[e] = pack16<F16>(v[2 * e], v[2 * e + 1]);
            *reinterpret_cast<uint4*>(sP + sw128_chunk(ri, jh / 8)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(sP + sw128_chunk(ri, jh / 8 + 1)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
      tc_fence_before();
      named_sync(kBarLocal, NT);
      // (4) T = (I + A)^-1
      solve_unit_lower(sA, sT, sX, at, kBarLocal);
      // (5) T diag(beta gam rk) -> bf16, T diag(beta) -> hi + lo (K-major rows i; 16 columns
      //     per thread)
      {
        const int ri = at >> 2, qd = at & 3;
        uint8_t* lw = S.wk() + WK_LW;
        uint8_t* luh = S.wk() + WK_LUHI;
        uint8_t* lul = S.wk() + WK_LULO;
        const float* trw = sT + ri * kAS;
        const float vmul = U.zero_v ? 0.f : 1.f;  // split-K transition maps run with v = 0
        // every shared-memory read before the first store (the stores could alias them)
        float tv[16], fv[16], bv[16];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int j0 = (2 * qd + h2) * 8;
#pragma unroll
          for (int e4 = 0; e4 < 8; e4 += 4) {
            const float4 ta = *reinterpret_cast<const float4*>(trw + j0 + e4);
            const float4 fa = *reinterpret_cast<const float4*>(sF1 + j0 + e4);
            const float4 ba = *reinterpret_cast<const float4*>(gbeta + j0 + e4);
            const int o = 8 * h2 + e4;
            tv[o] = ta.x; tv[o + 1] = ta.y; tv[o + 2] = ta.z; tv[o + 3] = ta.w;
            fv[o] = fa.x; fv[o + 1] = fa.y; fv[o + 2] = fa.z; fv[o + 3] = fa.w;
            bv[o] = vmul * ba.x; bv[o + 1] = vmul * ba.y; bv[o + 2] = vmul * ba.z; bv[o + 3] = vmul * ba.w;
          }
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int ch = 2 * qd + h2;
          uint32_t ww[4], wh[4], wl[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int o = 8 * h2 + 2 * e;
            const float t0v = tv[o], t1v = tv[o + 1];
            ww[e] = pack16<F16>(t0v * fv[o], t1v * fv[o + 1]);
            split16<F16>(t0v * bv[o], t1v * bv[o + 1], wh[e], wl[e]);
          }
          const uint32_t o = sw128_chunk(ri, ch);
          *reinterpret_cast<uint4*>(lw + o) = make_uint4(ww[0], ww[1], ww[2], ww[3]);
          *reinterpret_cast<uint4*>(luh + o) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
          *reinterpret_cast<uint4*>(lul + o) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(kBarLocal, NT);
      if (at == 0 && !(p.hold_local_ready && k == 0)) mbar_arrive(&bars->l_ready);
    }
  }
  if (!ok && at == 0) raise_abort(p, bars);
}

// Columns c0..c0+31 of row r of a unit's incoming state.
__device__ __forceinline__ void unit_state_in(const PrefillParams& p, int in_kind, int64_t in_ws, int64_t pool_off,
                                              int r, int c0, float (&v)[32]) {
  if (in_kind == kInPool && p.s_in) {
    load_state_chunk(p.s_in, p.sin_dtype, pool_off, c0, v);
  } else if (in_kind == kInWs) {
    load_state_chunk(p.ws, kF32, in_ws * (kHeadDim * kHeadDim) + (int64_t)r * kHeadDim, c0, v);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = (in_kind == kInIdentity && c0 + j == r) ? 1.f : 0.f;
  }
}
// Columns c0..c0+31 of row r of a unit's outgoing state.
__device__ __forceinline__ void unit_state_out(const PrefillParams& p, int out_kind, int64_t out_ws,
                                               int64_t pool_off, int r, int c0, const float* v) {
  if (out_kind == kOutPool) {
    if (p.s_out) store_state_chunk(p.s_out, p.sout_dtype, pool_off, c0, v);
  } else if (out_kind == kOutWs) {
    store_state_chunk(p.ws, kF32, out_ws * (kHeadDim * kHeadDim) + (int64_t)r * kHeadDim, c0, v);
  }
}

// The chain group's per-unit state work, out of line (it runs once per unit and would
// otherwise crowd the per-chunk code out of the instruction caches).
// Empty unit: the outgoing state is the incoming one.
__device__ __noinline__ void chain_state_copy(const PrefillParams& p, int in_kind, int64_t in_ws, int64_t sin_off,
                                              int out_kind, int64_t out_ws, int64_t sout_off, int r) {
#pragma unroll 1
  for (int c0 = 0; c0 < 128; c0 += 32) {
    float v32[32];
    unit_state_in(p, in_kind, in_ws, sin_off, r, c0, v32);
    unit_state_out(p, out_kind, out_ws, sout_off, r, c0, v32);
  }
}
// Incoming state row r: gl * S -> TMEM S and S -> the bf16 A-operand copy.
template <bool F16>
__device__ __noinline__ void chain_state_load(const PrefillParams& p, int in_kind, int64_t in_ws, int64_t sin_off,
                                              int r, uint32_t trow, float gl) {
  if (in_kind == kInPool && p.s_in && p.sin_dtype != kF32) {
    // 16-bit pool: 64 columns (8 x 16 B) in flight at once, two round trips per row
    const bool h16 = p.sin_dtype == kF16;
#pragma unroll 1
    for (int c64 = 0; c64 < 128; c64 += 64) {
      const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.s_in) + sin_off + c64);
      uint4 raw[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) raw[c] = __ldg(q + c);
#pragma unroll
      for (int cc = 0; cc < 64; cc += 32) {
        uint32_t rr[32], b16[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 x = raw[cc / 8 + c];
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = h16 ? __half22float2(*reinterpret_cast<const __half2*>(&w[e]))
                                 : __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
            b16[4 * c + e] = pack16<F16>(f.x, f.y);
            rr[8 * c + 2 * e] = __float_as_uint(f.x * gl);
            rr[8 * c + 2 * e + 1] = __float_as_uint(f.y * gl);
          }
        }
        tmem_st32(trow + TM_S + c64 + cc, rr);
        tmem_st16(trow + TM_SB + (c64 + cc) / 2, b16);
      }
    }
    tmem_st_wait();
    return;
  }
#pragma unroll 1
  for (int c0 = 0; c0 < 128; c0 += 32) {
    float v32[32];
    unit_state_in(p, in_kind, in_ws, sin_off, r, c0, v32);
    uint32_t rr[32], b16[16];
#pragma unroll
    for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(v32[j] * gl);
    tmem_st32(trow + TM_S + c0, rr);
#pragma unroll
    for (int j = 0; j < 16; ++j) b16[j] = pack16<F16>(v32[2 * j], v32[2 * j + 1]);
    tmem_st16(trow + TM_SB + c0 / 2, b16);
  }
  tmem_st_wait();
}
// Final state row r: TMEM S -> the unit's destination.
__device__ __noinline__ void chain_state_store(const PrefillParams& p, int out_kind, int64_t out_ws, int64_t sout_off,
                                               int r, uint32_t trow) {
#pragma unroll 1
  for (int c0 = 0; c0 < 128; c0 += 32) {
    uint32_t rr[32];
    tmem_ld32(trow + TM_S + c0, rr);
    tmem_ld_wait();
    float v32[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v32[j] = __uint_as_float(rr[j]);
    unit_state_out(p, out_kind, out_ws, sout_off, r, c0, v32);
  }
}
// Final state of the unit into a 16-bit pool with a tensor map: columns 0-63 through the
// K-copy slot `kc` of the unit's last chunk (free once the state-update MMA has read it;
// the caller holds its release to the producer) and columns 64-127 through the output
// stage, each written by one TMA store (rows of 128 B, 128B-swizzled).  All 128 chain
// threads; thread bt == 0 issues the stores.
__device__ __noinline__ void chain_state_store_tma(const PrefillParams& p, uint8_t* kc, uint8_t* stage, int r, int bt,
                                                   uint32_t trow, int h, int64_t slot) {
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    uint8_t* buf = hh ? stage : kc;
    if (hh == 1) {
      if (bt == 0) bulk_wait_read_but_newest();  // the chunk's output tile has left the stage
      named_sync(kBarChain, 128);
    }
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t rr[32];
      tmem_ld32(trow + TM_S + 64 * hh + c0, rr);
      tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(rr[8 * q + 2 * e]), hi = __uint_as_float(rr[8 * q + 2 * e + 1]);
          pk[e] = p.sout_dtype == kF16 ? pack_f16(lo, hi) : pack_bf16(lo, hi);
        }
        *reinterpret_cast<uint4*>(buf + sw128_chunk(r, c0 / 8 + q)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    fence_proxy_async_smem();
    named_sync(kBarChain, 128);
    if (bt == 0) {
      tma_store_4d(&p.tm_sout, buf, 64 * hh, 0, h, (int)slot);
      bulk_commit();
    }
  }
}
// Incoming state of a unit from a 16-bit pool with a tensor map: columns 0-63 into the
// held K-copy slot `kc`, columns 64-127 into the output stage, both by TMA at once (after
// the stores that last read those buffers); then row r: gl * S -> TMEM S and S -> the
// 16-bit copy, as chain_state_load.  Gives the K-copy slot back to the producer.  Returns
// false on a timeout (the loads have then been waited for with the full bound).
template <bool F16>
__device__ __noinline__ bool chain_state_load_tma(const PrefillParams& p, Bars* bars, uint8_t* kc, int kc_slot,
                                                  uint8_t* stage, int r, int bt, uint32_t trow, float gl, int h,
                                                  int64_t slot, uint32_t parity) {
  if (bt == 0) {
    bulk_wait_read_all();  // the final-state stores of the previous unit have read both buffers
    mbar_arrive_expect_tx(&bars->st_full, 2 * 16384);
    tma_load_4d(kc, &p.tm_sin, &bars->st_full, 0, 0, h, (int)slot);
    tma_load_4d(stage, &p.tm_sin, &bars->st_full, 64, 0, h, (int)slot);
  }
  const bool w = mbar_wait(&bars->st_full, parity, p.wait_ns);
  if (!named_sync_and(kBarChain, 128, w)) {
    if (bt == 0) mbar_wait(&bars->st_full, parity, kWaitLimitNs);  // the loads land before smem goes away
    return false;
  }
  const bool h16 = p.sin_dtype == kF16;
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    const uint8_t* buf = hh ? stage : kc;
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t rr[32], b16[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 x = *reinterpret_cast<const uint4*>(buf + sw128_chunk(r, c0 / 8 + q));
        const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = h16 ? __half22float2(*reinterpret_cast<const __half2*>(&wv[e]))
                               : __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[e]));
          b16[4 * q + e] = pack16<F16>(f.x, f.y);
          rr[8 * q + 2 * e] = __float_as_uint(f.x * gl);
          rr[8 * q + 2 * e + 1] = __float_as_uint(f.y * gl);
        }
      }
      tmem_st32(trow + TM_S + 64 * hh + c0, rr);
      tmem_st16(trow + TM_SB + (64 * hh + c0) / 2, b16);
    }
  }
  tmem_st_wait();
  fence_proxy_async_smem();  // these reads of the K-copy slot before the producer's next TMA into it
  named_sync(kBarChain, 128);
  if (bt == 0) mbar_arrive(&bars->empty_kc[kc_slot]);
  return true;
}
// Mid-sequence checkpoint: state row r (TMEM S, the state after the chunk) -> f32
// checkpoint block m of sequence n, head h.
__device__ __noinline__ void chain_ckpt_store(const PrefillParams& p, int n, int h, int m, int r, uint32_t trow) {
  float* dst = p.ck + (int64_t)n * p.ck_seq + (int64_t)m * p.ck_idx + (int64_t)h * p.ck_head + (int64_t)r * kHeadDim;
#pragma unroll 1
  for (int c0 = 0; c0 < 128; c0 += 32) {
    uint32_t rr[32];
    tmem_ld32(trow + TM_S + c0, rr);
    tmem_ld_wait();
    float4* d4 = reinterpret_cast<float4*>(dst + c0);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      d4[j] = make_float4(__uint_as_float(rr[4 * j]), __uint_as_float(rr[4 * j + 1]), __uint_as_float(rr[4 * j + 2]),
                          __uint_as_float(rr[4 * j + 3]));
  }
}

// ------------------------------------------------------------ warps 11-14: chain epilogues
template <bool F16>
__device__ __forceinline__ void run_chain_wg(const PrefillParams& p, const Smem S, uint32_t tmem, int warp, int lane) {
  Bars* bars = S.bars;
  const int bt = threadIdx.x - 32 * kWgChain;  // 0..127
  const int r = 32 * (warp & 3) + lane;        // value row v this thread owns
  const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  const int n_items = cta_items(p);
  int i = 0;
  bool ok = true;
  int jr = 0;  // units of this CTA so far
  int kc_held = -1;    // K-copy slot whose release waits for the next unit's state load
  uint32_t n_sld = 0;  // incoming states loaded by TMA
  for (int64_t u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++jr) {
    // the unit's record, from the producer; the previous unit's slot goes back to it (every
    // chain thread is past that unit once this barrier completes)
    const int rs = jr % kRecSlots;
    const bool wr = mbar_wait(&bars->rec_full[rs], (jr / kRecSlots) & 1, p.wait_ns);
    ok = named_sync_and(kBarChain, 128, wr && !aborted(bars));
    if (!ok) break;
    if (bt == 0 && jr > 0) mbar_arrive(&bars->rec_empty[(jr - 1) % kRecSlots]);
    const Unit& U = *S.rec(rs);
    const bool tma_in = kc_held >= 0 && !U.idle && !U.err && U.nch > 0 && U.in_kind == kInPool && p.s_in && p.sin_tma;
    if (kc_held >= 0 && !tma_in) {  // no TMA load to stage through the held slot: give it back
      if (bt == 0) {
        bulk_wait_read_all();
        mbar_arrive(&bars->empty_kc[kc_held]);
      }
      kc_held = -1;
    }
    if (U.idle) continue;
    if (U.err) {
      if (bt == 0) set_error(p.dev_err, U.err);
      continue;
    }
    const int64_t sin_off = p.s_in ? U.slot * p.sin_slot + (int64_t)U.h * p.sin_head + (int64_t)r * kHeadDim : 0;
    const int64_t sout_off = p.s_out ? U.slot * p.sout_slot + (int64_t)U.h * p.sout_head + (int64_t)r * kHeadDim : 0;
    if (U.nch == 0) {  // empty sequence (or segment): the final state is the initial state
      chain_state_copy(p, U.in_kind, U.in_ws, sin_off, U.out_kind, U.out_ws, sout_off, r);
      continue;
    }
    {  // initial state: S * gam_last(first chunk) -> TMEM S, S -> bf16 copy (A operand).  The
       // gates of every item after the CTA's first are awaited by the previous item's second
       // epilogue: each phase of gates_ready is consumed before the accumulator slot that
       // lets the chunk-local group run two items further is released.
      bool w = i > 0 || mbar_wait(&bars->gates_ready[0], 0, p.wait_ns);
      ok = named_sync_and(kBarChain, 128, w && !aborted(bars));
      if (!ok) break;
      if (tma_in) {
        ok = chain_state_load_tma<F16>(p, bars, S.KC(kc_held), kc_held, S.stage(), r, bt, trow,
                                       S.vmisc(i % kVecSlots)[0], U.h, U.slot, n_sld & 1);
        ++n_sld;
        kc_held = -1;
        if (!ok) break;
      } else {
        chain_state_load<F16>(p, U.in_kind, U.in_ws, sin_off, r, trow, S.vmisc(i % kVecSlots)[0]);
      }
      tc_fence_before();
      named_sync(kBarChain, 128);
      if (bt == 0) mbar_arrive(&bars->s_ready);
    }
    // the fields every chunk reads, in registers (the record stays in shared memory)
    const int64_t ubos = U.bos, ueos = U.eos;
    const int unch = U.nch, uh = U.h;
    const bool uwo = U.write_out;
    for (int c = 0; c < unch; ++c, ++i) {
      const int s = i & 1;
      const bool last = (c + 1 == unch);
      const int64_t t0 = ubos + (int64_t)c * kChunk;
      const int nvalid = (ueos - t0 < kChunk) ? (int)(ueos - t0) : kChunk;
      const uint32_t acc = trow + TM_ACC + s * 128;
      // ---- epilogue 1: Vn (fp32) -> bf16 Vn and Vd = Vn diag(d rk) hi / lo, O1 -> -gam O1
      bool w = mbar_wait(&bars->c1_done, i & 1, p.wait_ns);
      ok = named_sync_and(kBarChain, 128, w);
      if (!ok) break;
      tc_fence_after();
      {
        // Vn (fp32, columns 0-63) -> three bf16 operands of 32 columns each: Vn itself into
        // columns 0-31, Vd hi into the Vd hi columns and Vd lo into the S_bf columns (S_bf is
        // dead until epilogue 2), 16 Vn columns at a time.
        const float* dk = S.vdk(i % kVecSlots);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t raw[16], pn[8], ph[8], pl[8];
          tmem_ld16(acc + 16 * q, raw);
          float dq[16];
#pragma unroll
          for (int j4 = 0; j4 < 16; j4 += 4) {
            const float4 d4 = *reinterpret_cast<const float4*>(dk + 16 * q + j4);
            dq[j4] = d4.x; dq[j4 + 1] = d4.y; dq[j4 + 2] = d4.z; dq[j4 + 3] = d4.w;
          }
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float a = __uint_as_float(raw[2 * j]), b = __uint_as_float(raw[2 * j + 1]);
            pn[j] = pack16<F16>(a, b);
            float x0 = a, x1 = b;
            mul2(x0, x1, dq[2 * j], dq[2 * j + 1]);
            split16<F16>(x0, x1, ph[j], pl[j]);
          }
          tmem_st8(acc + 8 * q, pn);             // Vn as bf16 pairs: A operand of O += Vn P^T
          tmem_st8(trow + TM_VDH + 8 * q, ph);   // Vd hi and lo: A operands of the state update
          tmem_st8(trow + TM_SB + 8 * q, pl);
        }
        uint32_t rr[32];
        const float* gam = S.vgam(i % kVecSlots);
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
          tmem_ld32(acc + 64 + c0, rr);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float x0 = __uint_as_float(rr[j]), x1 = __uint_as_float(rr[j + 1]);
            mul2(x0, x1, -gam[c0 + j], -gam[c0 + j + 1]);
            rr[j] = __float_as_uint(x0);
            rr[j + 1] = __float_as_uint(x1);
          }
          tmem_st32(acc + 64 + c0, rr);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      named_sync(kBarChain, 128);
      if (bt == 0) mbar_arrive(&bars->vd_ready);
      // ---- epilogue 2: the output tile (its TMA store left in flight), which releases the
      //      accumulator slot; then S -> bf16 copy and gam_last(next) S, or the final state
      const bool c2ok = mbar_wait(&bars->c2_done, i & 1, p.wait_ns);
      w = c2ok;
      if (w && i + 1 < n_items) w = mbar_wait(&bars->gates_ready[(i + 1) & 1], ((i + 1) >> 1) & 1, p.wait_ns);
      const bool hold_kc = last && U.out_kind == kOutPool && p.s_out && p.sout_tma;  // staging buffer
      if (bt == 0) {
        if (c2ok && !hold_kc) mbar_arrive(&bars->empty_kc[s]);  // the state-update MMA has read its K copy
        bulk_wait_read_all();                                   // the previous output tile has left the stage
      }
      ok = named_sync_and(kBarChain, 128, w);
      if (!ok) break;
      tc_fence_after();
      if (p.ck && uwo && nvalid == kChunk) {  // a checkpoint after this chunk?
        const int ca = U.c_off + c + 1;                  // chunks of the sequence done
        if (ca % p.ck_every == 0 && ca / p.ck_every <= p.ck_count)
          chain_ckpt_store(p, U.n, U.h, ca / p.ck_every - 1, r, trow);
      }
      if (uwo) {
        // the 64 x 128 tile, read as m16n8 fragments (16 value rows at a time) and stored
        // transposed by stmatrix into token rows of the two 128B-swizzled halves of the stage
        // (values 0-63 | 64-127), for two TMA stores (or, in a partial last chunk, a copy of
        // its valid rows)
        const uint32_t stage = smem_u32(S.stage());
        const float* pq = S.vrq(i % kVecSlots);
        const int mi = lane >> 3, jr = lane & 7;  // stored matrix and row this lane addresses
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {  // 16 value rows x 32 tokens per step
          const int dv0 = 32 * (warp & 3) + 16 * (q4 >> 1), tk0 = 32 * (q4 & 1);
          uint32_t rr[16];
          tmem_ld16x256_x4(tmem + ((uint32_t)dv0 << 16) + TM_ACC + s * 128 + 64 + tk0, rr);
          tmem_ld_wait();
          const int dv = dv0 + 8 * (mi & 1);  // first value row of the lane's stored matrix
          const uint32_t hb = stage + (uint32_t)(dv >> 6) * 8192, cc = (uint32_t)((dv & 63) >> 3);
#pragma unroll
          for (int gp = 0; gp < 2; ++gp) {
            const int tok = tk0 + 16 * gp + 8 * (mi >> 1) + jr;
            const uint32_t* x = rr + 8 * gp;
            // this lane's token columns: tk0 + 16 gp + 2 (lane % 4) + {0, 1}, and + 8
            const float2 f0 = *reinterpret_cast<const float2*>(pq + tk0 + 16 * gp + 2 * (lane & 3));
            const float2 f1 = *reinterpret_cast<const float2*>(pq + tk0 + 16 * gp + 8 + 2 * (lane & 3));
            stmatrix_x4_trans(hb + (uint32_t)tok * 128 + ((cc ^ (uint32_t)jr) << 4),
                              pack16<F16>(f0.x * __uint_as_float(x[0]), f0.y * __uint_as_float(x[1])),
                              pack16<F16>(f0.x * __uint_as_float(x[2]), f0.y * __uint_as_float(x[3])),
                              pack16<F16>(f1.x * __uint_as_float(x[4]), f1.y * __uint_as_float(x[5])),
                              pack16<F16>(f1.x * __uint_as_float(x[6]), f1.y * __uint_as_float(x[7])));
          }
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      named_sync(kBarChain, 128);
      if (bt == 0) {
        mbar_arrive(&bars->acc_free[s]);
        if (uwo && nvalid == kChunk) {
          tma_store_3d(&p.tm_o, S.stage(), 0, uh, (int)t0);
          tma_store_3d(&p.tm_o, S.stage() + 8192, 64, uh, (int)t0);
          bulk_commit();
        }
      }
      if (uwo && nvalid < kChunk) {
        // partial last chunk: its nvalid token rows (16 x 16 bytes each) from the stage
        uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + t0 * p.o_st + (int64_t)uh * p.o_sh;
        for (int e = bt; e < nvalid * 16; e += 128) {
          const int row = e >> 4, hc = (e >> 3) & 1, cq = e & 7;
          const uint4 x = *reinterpret_cast<const uint4*>(S.stage() + hc * 8192 + row * 128 + ((cq ^ (row & 7)) << 4));
          *reinterpret_cast<uint4*>(orow + (int64_t)row * p.o_st + hc * 64 + cq * 8) = x;
        }
      }
      if (hold_kc) {
        chain_state_store_tma(p, S.KC(s), S.stage(), r, bt, trow, uh, U.slot);
        kc_held = s;
      } else if (last) {
        chain_state_store(p, U.out_kind, U.out_ws, sout_off, r, trow);
      } else {
        uint32_t rr[32];
        const float gl = S.vmisc((i + 1) % kVecSlots)[0];
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          tmem_ld32(trow + TM_S + c0, rr);
          tmem_ld_wait();
          uint32_t b16[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) b16[j] = pack16<F16>(__uint_as_float(rr[2 * j]), __uint_as_float(rr[2 * j + 1]));
          tmem_st16(trow + TM_SB + c0 / 2, b16);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float x0 = __uint_as_float(rr[j]), x1 = __uint_as_float(rr[j + 1]);
            mul2(x0, x1, gl, gl);
            rr[j] = __float_as_uint(x0);
            rr[j + 1] = __float_as_uint(x1);
          }
          tmem_st32(trow + TM_S + c0, rr);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      named_sync(kBarChain, 128);
      if (bt == 0 && !last) mbar_arrive(&bars->s_ready);
    }
  }
  if (bt == 0) bulk_wait_read_all();  // the last tile has left the stage before the CTA exits
  if (kc_held >= 0 && bt == 0) mbar_arrive(&bars->empty_kc[kc_held]);
  if (!ok && bt == 0) raise_abort(p, bars);
}

// ------------------------------------------------------------ the kernel
template <bool F16>
__global__ void __launch_bounds__(kThreads, 1) gdn_prefill_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem S;
  S.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  S.bars = reinterpret_cast<Bars*>(S.base + OFF_BAR);
  Bars* bars = S.bars;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    uint64_t* b = reinterpret_cast<uint64_t*>(bars);
    const int nbars = (int)(offsetof(Bars, tmem_base) / sizeof(uint64_t));
    for (int k = 0; k < nbars; ++k) mbar_init(&b[k], 1);
    bars->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }
  if (warp == kWarpProducer) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kWarpProducer) run_producer(p, S, lane);
  else if (warp == kWarpMmaLocal) run_mma_local<F16>(p, S, tmem, lane == 0);
  else if (warp == kWarpMmaChain) run_mma_chain<F16>(p, S, tmem, lane == 0);
  else if (warp < kWgChain) run_local_wg<F16>(p, S, tmem, warp, lane);
  else run_chain_wg<F16>(p, S, tmem, warp, lane);

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpProducer) tmem_dealloc(tmem, kTmemCols);
}


// ------------------------------------------------------------ split-K state fix-up
// For every (sequence, head) of a split launch, walk the segments in order:
// S_{p+1} = S_p M_p + N_p (p = 1..P-2), all fp32, reading S_1 and the segment maps
// that the first pass left in the workspace and writing S_2..S_{P-1} back.  Row r of
// S_{p+1} needs only row r of S_p, so each (sequence, head) is shared by kFixParts CTAs
// of kFixRows rows each, every one walking all the segments for its rows.
constexpr int kFixThreads = 256;
constexpr int kFixParts = 4;
constexpr int kFixRows = kHeadDim / kFixParts;  // 32: two rows x eight columns per thread
constexpr int kFixSStride = 132;  // padded fp32 row stride of the S rows in shared memory
constexpr size_t kFixSmemBytes = (size_t)(kFixRows * kFixSStride + kHeadDim * kHeadDim) * sizeof(float);

__global__ void __launch_bounds__(kFixThreads) gdn_split_fixup_kernel(float* ws, int P) {
  extern __shared__ float fx[];
  float* Ss = fx;                          // rows of S_p  [32][132]
  float* Ms = fx + kFixRows * kFixSStride;  // M_p          [128][128]
  constexpr int64_t kBlk = (int64_t)kHeadDim * kHeadDim;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;  // rows 2 ty, 2 ty + 1; columns 8 tx ..
  const int part = blockIdx.x % kFixParts;
  float* base = ws + (int64_t)(blockIdx.x / kFixParts) * split_ws_blocks(P) * kBlk;
  const int64_t r0 = (int64_t)part * kFixRows * kHeadDim;  // first element of this CTA's rows
  for (int e = 4 * tid; e < kFixRows * kHeadDim; e += 4 * kFixThreads) {
    const float4 v = *reinterpret_cast<const float4*>(base + r0 + e);
    *reinterpret_cast<float4*>(Ss + (e >> 7) * kFixSStride + (e & 127)) = v;
  }
#pragma unroll 1
  for (int sp = 1; sp <= P - 2; ++sp) {
    const float* M = base + (int64_t)(P - 1 + sp - 1) * kBlk;
    const float* Nn = base + (int64_t)(2 * P - 3 + sp - 1) * kBlk + r0;
    float* Snext = base + (int64_t)sp * kBlk + r0;
    for (int e = 4 * tid; e < kBlk; e += 4 * kFixThreads)
      *reinterpret_cast<float4*>(Ms + e) = *reinterpret_cast<const float4*>(M + e);
    __syncthreads();
    float acc[2][8];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
#pragma unroll 8
    for (int kk = 0; kk < kHeadDim; ++kk) {
      const float4 b0 = *reinterpret_cast<const float4*>(Ms + kk * kHeadDim + 8 * tx);
      const float4 b1 = *reinterpret_cast<const float4*>(Ms + kk * kHeadDim + 8 * tx + 4);
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const float sv = Ss[(2 * ty + a) * kFixSStride + kk];
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(sv, bv[b], acc[a][b]);
      }
    }
    __syncthreads();  // every read of S_p and M_p is done
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int row = 2 * ty + a;
      const float4 n0 = *reinterpret_cast<const float4*>(Nn + row * kHeadDim + 8 * tx);
      const float4 n1 = *reinterpret_cast<const float4*>(Nn + row * kHeadDim + 8 * tx + 4);
      const float4 o0 = make_float4(acc[a][0] + n0.x, acc[a][1] + n0.y, acc[a][2] + n0.z, acc[a][3] + n0.w);
      const float4 o1 = make_float4(acc[a][4] + n1.x, acc[a][5] + n1.y, acc[a][6] + n1.z, acc[a][7] + n1.w);
      *reinterpret_cast<float4*>(Snext + row * kHeadDim + 8 * tx) = o0;
      *reinterpret_cast<float4*>(Snext + row * kHeadDim + 8 * tx + 4) = o1;
      *reinterpret_cast<float4*>(Ss + row * kFixSStride + 8 * tx) = o0;
      *reinterpret_cast<float4*>(Ss + row * kFixSStride + 8 * tx + 4) = o1;
    }
    __syncthreads();
  }
}

struct LaunchConfig {
  int device = -1;
  int num_sms = 0;
  int generation = -1;
};
thread_local LaunchConfig t_cfg;
std::atomic<int> g_config_generation{0};

cudaError_t configure_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int gen = g_config_generation.load(std::memory_order_acquire);
  if (t_cfg.device == dev && t_cfg.generation == gen) return cudaSuccess;
  e = cudaFuncSetAttribute(gdn_prefill_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gdn_prefill_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gdn_split_fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFixSmemBytes);
  int sms = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  t_cfg.device = dev;
  t_cfg.num_sms = sms;
  t_cfg.generation = gen;
  return cudaSuccess;
}

}  // namespace

int launch_config_generation() { return g_config_generation.load(std::memory_order_acquire); }

void invalidate_launch_config() { g_config_generation.fetch_add(1, std::memory_order_acq_rel); }

// The scratch of the allocation-free entry point lives in the module's static
// device memory, so using it needs no allocation call.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocHeaderBytes + kNoAllocWorkspaceBytes];

cudaError_t noalloc_scratch(void** base) { return cudaGetSymbolAddress(base, g_noalloc_scratch); }

size_t prefill_smem_bytes() { return kSmemBytes; }

int device_sm_count() { return configure_device() == cudaSuccess ? t_cfg.num_sms : 0; }

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream) {
  cudaError_t e = configure_device();
  if (e != cudaSuccess) return e;
  if (p.n_units <= 0) return cudaSuccess;
  const unsigned grid = p.grid > 0 ? (unsigned)p.grid
                                   : (unsigned)(p.n_units < t_cfg.num_sms ? p.n_units : t_cfg.num_sms);
  if (p.op_f16) gdn_prefill_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(p);
  else gdn_prefill_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_split_fixup(const PrefillParams& p, cudaStream_t stream) {
  cudaError_t e = configure_device();
  if (e != cudaSuccess) return e;
  const int64_t units = (int64_t)p.N * p.H;
  if (p.splits < 3 || units <= 0) return cudaSuccess;
  gdn_split_fixup_kernel<<<(unsigned)(units * kFixParts), kFixThreads, kFixSmemBytes, stream>>>(p.ws, p.splits);
  return cudaGetLastError();
}

}  // namespace gdn
