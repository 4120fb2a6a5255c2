// Internal interface between the C-ABI host code (api.cpp) and the kernels
// (prefill.cu).  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime_api.h>
#include <stdint.h>

namespace gdn {

constexpr int kHeadDim = 128;  // Dk = Dv = 128 (the only head size the operation defines)
constexpr int kChunk = 64;     // tokens per chunk tile

enum DType : int32_t { kF32 = 0, kBF16 = 1, kF16 = 2, kI32 = 3, kI64 = 4 };

// Everything one launch needs.  Passed by value as a __grid_constant__ kernel
// parameter, so the TMA descriptors live in parameter space for the launch only.
struct PrefillParams {
  CUtensorMap tm_q;  // [T, H_qk, 128] bf16, box (64 dk, 1 head, 64 tokens), 128B swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;  // [T, H_v, 128]
  CUtensorMap tm_o;  // output [T, H, 128] bf16, box (64 dv, 1 head, 64 tokens), 128B swizzle (stores)
  CUtensorMap tm_sout;  // 16-bit output-state pool [slots, H, 128, 128], box (64 cols, 128 rows, 1, 1),
                        // 128B swizzle (stores); valid when sout_tma != 0
  CUtensorMap tm_sin;   // 16-bit input-state pool, the same boxes (loads); valid when sin_tma != 0
  const void* g;     // [T, H] or null; strides in elements
  int64_t g_st, g_sh;
  const void* beta;
  int64_t b_st, b_sh;
  const void* s_in;  // [slots, H, 128, 128] or null
  int64_t sin_slot, sin_head, sin_slots;
  void* s_out;       // [slots, H, 128, 128] or null
  int64_t sout_slot, sout_head, sout_slots;
  const void* state_idx;  // [N] or null
  const void* cu;         // [N + 1]
  void* out;              // [T, H, 128] bf16
  int64_t o_st, o_sh;
  int32_t* dev_err;       // device error word (GDN_DEVERR_* bits)
  int64_t T;
  int32_t N, H, H_qk, H_v;
  int32_t g_dtype, b_dtype, sin_dtype, sout_dtype, idx_dtype, cu_dtype;
  float scale;
  int32_t l2norm;
  int32_t op_f16;  // q/k/v/output (and every tensor-core operand) fp16 instead of bf16
  // split-K: mode 0 walks whole sequences; mode 1 (pass 1) walks, per (sequence, head),
  // segment 0 and the affine maps (M_p, N_p) of the middle segments; mode 2 (pass 2)
  // walks segments 1..P-1 from their fixed-up incoming states.
  int32_t mode;
  int32_t splits;          // P, segments per sequence (modes 1, 2)
  // segment p of a sequence of C chunks holds chunks [C seg_num[p] / seg_den,
  // C seg_num[p + 1] / seg_den) (seg_num[0] = 0, seg_num[P] = seg_den)
  int32_t seg_num[9];
  int32_t seg_den;
  // Unit order of a split launch (modes 1, 2).  n_runs = 0: per (sequence, head) its
  // units in a row (2P - 3 in mode 1, P - 1 in mode 2).  Otherwise the launch's units are
  // cut into n_runs runs, run r covering units [runs[r - 1].u_end, runs[r].u_end) (from 0
  // for r = 0); unit u of a run stands for j = first + (u - start of the run):
  //   kind >= 0        (sequence, head) j, unit kind `kind` (mode 1: 0 = segment 0, p in
  //                    1..P-2 = M_p, P - 2 + p = N_p; mode 2: segment kind + 1);
  //   kind == kRunMaps the j-th map walk: (sequence, head) j / (2P - 4), kind 1 + j % (2P - 4);
  //   kind == kRunIdle no unit (the CTA that meets it goes on to its next index).
  // CTA c walks units c, c + grid, c + 2 grid, ..., so a plan places each unit on a CTA.
  struct UnitRun {
    int32_t u_end, first, kind, pad_;
  };
  static constexpr int32_t kRunMaps = -1, kRunIdle = -2;
  static constexpr int kMaxRuns = 8;
  int32_t n_runs;
  UnitRun runs[kMaxRuns];
  int32_t grid;            // CTAs of the launch (0: min(n_units, SMs))
  float* ws;               // fp32 [N][H][3P - 5][128][128] (modes 1, 2)
  int64_t n_units;         // units this launch walks
  // mid-sequence checkpoints (null: none): f32 blocks of 128 x 128, checkpoint m of
  // sequence n and head h at ck + n ck_seq + m ck_idx + h ck_head (elements); it is the
  // state after (m + 1) * ck_every chunks
  float* ck;
  int64_t ck_seq, ck_idx, ck_head;
  int32_t ck_count, ck_every;
  // bound of every on-chip wait (a timeout sets GDN_DEVERR_TIMEOUT and ends the CTA's
  // work), and a testing aid: nonzero makes the chunk-local group withhold its first
  // "operands ready" arrival, so that the wait for it runs out
  uint64_t wait_ns;
  int32_t hold_local_ready;
  int32_t sout_tma;  // final states to the pool through tm_sout (16-bit pools whose strides allow it)
  int32_t sin_tma;   // incoming states from the pool through tm_sin (likewise)
};

// Unit index u of a split launch (mode 1 or 2) -> its (sequence, head) index nh =
// n H + h and its kind, following the plan's runs (or the plain order without runs);
// false for an index that holds no unit.  Used by the kernel and by the host-side
// check of a plan.
__host__ __device__ inline bool split_unit(const PrefillParams& p, int64_t u, int32_t* nh, int32_t* kind) {
  const int P = p.splits;
  if (p.n_runs <= 0) {  // split launches hold fewer than 2^31 units: 32-bit divisions
    const uint32_t K = (uint32_t)(p.mode == 1 ? 2 * P - 3 : P - 1), u32 = (uint32_t)u, q = u32 / K;
    *nh = (int32_t)q;
    *kind = (int32_t)(u32 - q * K);
    return true;
  }
  int r = 0, start = 0;
  while (r + 1 < p.n_runs && u >= p.runs[r].u_end) start = p.runs[r++].u_end;
  const int32_t j = p.runs[r].first + (int32_t)(u - start), rk = p.runs[r].kind;
  if (rk == PrefillParams::kRunIdle) return false;
  if (rk == PrefillParams::kRunMaps) {
    const int32_t km = 2 * P - 4;
    *nh = j / km;
    *kind = 1 + (j - *nh * km);
  } else {
    *nh = j;
    *kind = rk;
  }
  return true;
}

// Blocks of 128 x 128 fp32 the split-K workspace holds per (sequence, head).
__host__ __device__ inline int64_t split_ws_blocks(int P) { return P >= 2 ? 3 * (int64_t)P - 5 : 0; }

// Dynamic shared memory the prefill kernel needs (bytes).
size_t prefill_smem_bytes();

// Enqueue the prefill on `stream`; returns the launch error (cudaSuccess if none).
cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream);

// Split-K state fix-up between the two passes: for every (sequence, head) and
// p = 1..P-2, S_{p+1} = S_p M_p + N_p in fp32 (workspace blocks).
cudaError_t launch_split_fixup(const PrefillParams& p, cudaStream_t stream);

// Streaming multiprocessors of the current device (cached).
int device_sm_count();

// Generation of the per-thread launch settings (kernel attributes, SM counts) that the
// launchers cache; gdn_shutdown bumps it so that every thread sets them up again (a
// device reset after the shutdown drops the attributes).
int launch_config_generation();
void invalidate_launch_config();

// Static scratch of the allocation-free entry point: a header (its first word is the
// device error word when the caller passes none) followed by the split-K workspace.
constexpr size_t kNoAllocHeaderBytes = 256;
constexpr size_t kNoAllocWorkspaceBytes = size_t(32) << 20;  // 512 state blocks of 64 KiB

// Device address of that scratch on the current device (cudaGetSymbolAddress).
cudaError_t noalloc_scratch(void** base);

}  // namespace gdn
