// C-ABI entry points of the chunked Gated Delta Rule prefill library: argument
// validation (fail closed, nothing launched on any error), default resolution,
// TMA descriptor encoding and the launch.  The argument contract is the one of
// flashinfer.cudnn.cudnn_chunk_gated_delta_rule (Parameters), restated in
// include/gdn.h.
#include "gdn.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "decode.h"
#include "prefill.h"

namespace {

thread_local char g_last_error[512] = "";

gdn_status_t fail(gdn_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

constexpr int kMaxDevices = 64;
struct DeviceState {
  bool ready = false;
  int32_t* dev_err = nullptr;  // device error word
  float* ws = nullptr;         // split-K workspace (grow-only, stream-ordered allocation)
  size_t ws_bytes = 0;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

size_t elem_size(int32_t dt) {
  switch (dt) {
    case GDN_F32: case GDN_I32: return 4;
    case GDN_BF16: case GDN_F16: return 2;
    case GDN_I64: return 8;
    default: return 0;
  }
}
const char* dt_name(int32_t dt) {
  switch (dt) {
    case GDN_F32: return "f32"; case GDN_BF16: return "bf16"; case GDN_F16: return "f16";
    case GDN_I32: return "i32"; case GDN_I64: return "i64"; default: return "?";
  }
}

// Byte range [lo, hi) a strided view can touch.
struct Range { uintptr_t lo, hi; };
Range byte_range(const gdn_tensor_t* t) {
  uintptr_t base = reinterpret_cast<uintptr_t>(t->data);
  int64_t span = 0;
  for (int i = 0; i < t->ndim; ++i) {
    if (t->shape[i] == 0) return {base, base};
    span += (t->shape[i] - 1) * t->stride[i];
  }
  return {base, base + (uintptr_t)((span + 1) * (int64_t)elem_size(t->dtype))};
}
bool overlaps(const gdn_tensor_t* a, const gdn_tensor_t* b) {
  if (!a || !b) return false;
  Range x = byte_range(a), y = byte_range(b);
  if (x.lo == x.hi || y.lo == y.hi) return false;
  return x.lo < y.hi && y.lo < x.hi;
}

gdn_status_t check_basic(const gdn_tensor_t* t, const char* name, int ndim) {
  if (!t) return fail(GDN_ERR_INVALID_ARGUMENT, "%s is required", name);
  if (t->ndim != ndim) return fail(GDN_ERR_INVALID_ARGUMENT, "%s must have %d dims, got %d", name, ndim, t->ndim);
  if (elem_size(t->dtype) == 0) return fail(GDN_ERR_INVALID_ARGUMENT, "%s has an unknown dtype %d", name, t->dtype);
  int64_t numel = 1;
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0) return fail(GDN_ERR_INVALID_ARGUMENT, "%s has a negative size", name);
    if (t->stride[i] < 0) return fail(GDN_ERR_INVALID_ARGUMENT, "%s has a negative stride", name);
    numel *= t->shape[i];
  }
  if (numel > 0 && !t->data) return fail(GDN_ERR_INVALID_ARGUMENT, "%s has a null data pointer", name);
  return GDN_OK;
}

gdn_status_t ensure_encode() {
  if (g_encode) return GDN_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
    return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable (%s)", cudaGetErrorString(e));
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return GDN_OK;
}

// q/k/v: [T, heads, 128] bf16 read in boxes of (64 dk, 1 head, 64 tokens), 128B swizzle.
gdn_status_t encode_qkv(CUtensorMap* m, const gdn_tensor_t* t, const char* name) {
  memset(m, 0, sizeof(*m));
  if (t->shape[0] == 0) return GDN_OK;  // no token will ever be loaded
  cuuint64_t dims[3] = {(cuuint64_t)t->shape[2], (cuuint64_t)t->shape[1], (cuuint64_t)t->shape[0]};
  cuuint64_t strides[2] = {(cuuint64_t)t->stride[1] * 2, (cuuint64_t)t->stride[0] * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, t->dtype == GDN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, t->data, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GDN_ERR_INVALID_ARGUMENT, "TMA descriptor for %s rejected (CUresult %d)", name, (int)r);
  return GDN_OK;
}

// output: [T, H, 128] bf16 written in boxes of (64 dv, 1 head, 64 tokens), 128B swizzle.
gdn_status_t encode_out(CUtensorMap* m, const gdn_tensor_t* t) {
  memset(m, 0, sizeof(*m));
  if (t->shape[0] == 0) return GDN_OK;
  cuuint64_t dims[3] = {(cuuint64_t)t->shape[2], (cuuint64_t)t->shape[1], (cuuint64_t)t->shape[0]};
  cuuint64_t strides[2] = {(cuuint64_t)t->stride[1] * 2, (cuuint64_t)t->stride[0] * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, t->dtype == GDN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, t->data, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GDN_ERR_INVALID_ARGUMENT, "TMA descriptor for output rejected (CUresult %d)", (int)r);
  return GDN_OK;
}

// 16-bit state pool [slots, H, 128, 128] moved in boxes of (64 cols, 128 rows, 1 head, 1
// slot), 128B swizzle; false when its strides rule a tensor map out (the kernel then
// moves rows with plain loads and stores).
bool encode_state_pool(CUtensorMap* m, const gdn_tensor_t* t) {
  memset(m, 0, sizeof(*m));
  if (t->dtype != GDN_BF16 && t->dtype != GDN_F16) return false;
  if ((t->stride[0] * 2) % 16 || (t->stride[1] * 2) % 16 || (reinterpret_cast<uintptr_t>(t->data) % 16)) return false;
  cuuint64_t dims[4] = {128, 128, (cuuint64_t)t->shape[1], (cuuint64_t)t->shape[0]};
  cuuint64_t strides[3] = {256, (cuuint64_t)t->stride[1] * 2, (cuuint64_t)t->stride[0] * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, t->dtype == GDN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                        t->data, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

gdn_status_t check_qkv(const gdn_tensor_t* t, const char* name) {
  gdn_status_t st = check_basic(t, name, 3);
  if (st != GDN_OK) return st;
  if (t->dtype != GDN_BF16 && t->dtype != GDN_F16)
    return fail(GDN_ERR_UNSUPPORTED, "%s must be bf16 or f16, got %s", name, dt_name(t->dtype));
  if (t->shape[2] != 128) return fail(GDN_ERR_UNSUPPORTED, "%s head_dim must be 128, got %lld", name, (long long)t->shape[2]);
  if (t->shape[1] < 1) return fail(GDN_ERR_INVALID_ARGUMENT, "%s needs at least one head", name);
  if (t->stride[2] != 1) return fail(GDN_ERR_INVALID_ARGUMENT, "%s innermost dim must be contiguous", name);
  if (t->shape[0] > 0) {
    if ((t->stride[0] % 8) || (t->stride[1] % 8) || t->stride[0] <= 0 || t->stride[1] <= 0)
      return fail(GDN_ERR_INVALID_ARGUMENT, "%s token/head strides must be positive multiples of 8 elements", name);
    if (reinterpret_cast<uintptr_t>(t->data) % 16) return fail(GDN_ERR_INVALID_ARGUMENT, "%s must be 16-byte aligned", name);
    if (t->shape[0] >= (int64_t(1) << 31) - 64) return fail(GDN_ERR_UNSUPPORTED, "%s has too many tokens", name);
  }
  return GDN_OK;
}

gdn_status_t check_gate(const gdn_tensor_t* t, const char* name, int64_t T, int64_t H, bool allow_f16) {
  if (!t) return GDN_OK;
  gdn_status_t st = check_basic(t, name, 2);
  if (st != GDN_OK) return st;
  if (!(t->dtype == GDN_F32 || t->dtype == GDN_BF16 || (allow_f16 && t->dtype == GDN_F16)))
    return fail(GDN_ERR_UNSUPPORTED, "%s dtype %s is not supported", name, dt_name(t->dtype));
  if (t->shape[0] != T || t->shape[1] != H)
    return fail(GDN_ERR_INVALID_ARGUMENT, "%s must be [T=%lld, H=%lld]", name, (long long)T, (long long)H);
  return GDN_OK;
}

gdn_status_t check_state(const gdn_tensor_t* t, const char* name, int64_t H) {
  if (!t) return GDN_OK;
  gdn_status_t st = check_basic(t, name, 4);
  if (st != GDN_OK) return st;
  if (t->dtype != GDN_F32 && t->dtype != GDN_BF16 && t->dtype != GDN_F16)
    return fail(GDN_ERR_UNSUPPORTED, "%s must be f32, bf16 or f16, got %s", name, dt_name(t->dtype));
  if (t->shape[1] != H || t->shape[2] != 128 || t->shape[3] != 128)
    return fail(GDN_ERR_INVALID_ARGUMENT, "%s must be [slots, H=%lld, 128, 128]", name, (long long)H);
  if (t->stride[3] != 1 || t->stride[2] != 128)
    return fail(GDN_ERR_INVALID_ARGUMENT, "%s inner 128 x 128 block must be contiguous (V-major)", name);
  const int64_t vec = 16 / (int64_t)elem_size(t->dtype);
  if ((t->stride[0] % vec) || (t->stride[1] % vec) || reinterpret_cast<uintptr_t>(t->data) % 16)
    return fail(GDN_ERR_INVALID_ARGUMENT, "%s slot/head strides must keep rows 16-byte aligned", name);
  return GDN_OK;
}

gdn_status_t check_index_vec(const gdn_tensor_t* t, const char* name, int64_t n) {
  gdn_status_t st = check_basic(t, name, 1);
  if (st != GDN_OK) return st;
  if (t->dtype != GDN_I32 && t->dtype != GDN_I64) return fail(GDN_ERR_UNSUPPORTED, "%s must be i32 or i64", name);
  if (n >= 0 && t->shape[0] != n) return fail(GDN_ERR_INVALID_ARGUMENT, "%s must have %lld entries", name, (long long)n);
  if (t->shape[0] > 1 && t->stride[0] != 1) return fail(GDN_ERR_INVALID_ARGUMENT, "%s must be contiguous", name);
  return GDN_OK;
}

// The device must be an sm_103 part with enough opt-in shared memory per block.
gdn_status_t check_device(int device) {
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
  if (prop.major != 10 || prop.minor != 3)
    return fail(GDN_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", device,
                prop.major, prop.minor);
  if (prop.sharedMemPerBlockOptin < gdn::prefill_smem_bytes())
    return fail(GDN_ERR_UNSUPPORTED, "device %d offers %zu B of shared memory per block, %zu needed", device,
                (size_t)prop.sharedMemPerBlockOptin, gdn::prefill_smem_bytes());
  return GDN_OK;
}

gdn_status_t init_device(int device) {
  if (device < 0 || device >= kMaxDevices) return fail(GDN_ERR_INVALID_ARGUMENT, "device %d out of range", device);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[device];
  if (d.ready) return GDN_OK;
  gdn_status_t st = check_device(device);
  if (st != GDN_OK) return st;
  cudaError_t e;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != device) cudaSetDevice(device);
  e = cudaMalloc(&d.dev_err, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(d.dev_err, 0, sizeof(int32_t));
  if (prev != device && prev >= 0) cudaSetDevice(prev);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "device error word: %s", cudaGetErrorString(e));
  st = ensure_encode();
  if (st != GDN_OK) return st;
  d.ready = true;
  return GDN_OK;
}

// Split-K plan of a call: P segments per sequence (1 = no split), their chunk
// boundaries (segment p = chunks [C num[p] / den, C num[p + 1] / den) of a C-chunk
// sequence), and the unit order and grid of each pass.
//
// Cost model, in walks of a whole sequence, with balanced lengths and U = N H units on a
// persistent grid of one CTA per SM (S SMs).  A middle segment costs three walks (its
// two maps in pass 1, its re-run in pass 2):
//  * uniform segments: pass 1 walks U (2P - 3) units of 1/P and pass 2 U (P - 1), in
//    ceil(units / S) rounds each: (ceil(U (2P - 3) / S) + ceil(U (P - 1) / S)) / P;
//  * P = 3 with segments of 1/2, 1/4, 1/4, when pass 1's 3U units exceed S by at most U:
//    the 3U - S CTAs that take two units are given two map walks of 1/4 each, so pass 1
//    takes 1/2 and pass 2 (2U units of 1/4) 1/4 per round;
//  * P = 4 with segments of R, 1, 1, 2 parts of R + 4, when U < S and 2U <= S: in pass 1,
//    U CTAs walk segment 0 (R parts) while the other m = S - U CTAs walk the 4U map walks
//    of one part each, R = ceil(4U / m) <= 3 to a CTA; in pass 2, U CTAs re-run segments
//    1 and 2 one after the other and U more re-run segment 3 (2 parts each):
//    (R + 2) / (R + 4).
// A plan is taken only when it saves at least a fifth and every segment keeps 8 chunks or
// more.
constexpr int kMaxSplits = 8;
constexpr size_t kMaxSplitWorkspace = size_t(4) << 30;
using UnitRun = gdn::PrefillParams::UnitRun;
constexpr int kMaxRuns = gdn::PrefillParams::kMaxRuns;

struct SplitPlan {
  int P = 1;
  int num[kMaxSplits + 1] = {0, 1};
  int den = 1;
  int n_runs[2] = {0, 0};  // unit order of pass 1 and pass 2 (0: per (sequence, head) in a row)
  UnitRun runs[2][kMaxRuns] = {};
  int64_t units[2] = {0, 0};
  int grid[2] = {0, 0};  // 0: min(units, S)

  void push(int pass, int64_t u_end, int64_t first, int32_t kind) {
    runs[pass][n_runs[pass]++] = UnitRun{(int32_t)u_end, (int32_t)first, kind, 0};
  }
};

SplitPlan uniform_plan(int P, int64_t U) {
  SplitPlan pl;
  pl.P = P;
  pl.den = P;
  for (int i = 0; i <= P; ++i) pl.num[i] = i;
  pl.units[0] = U * (2 * P - 3);
  pl.units[1] = U * (P - 1);
  return pl;
}

// P = 3, segments 1/2, 1/4, 1/4; x = 3U - S map walks lead the order of pass 1, so that
// the CTAs that take a second unit (c + S) take two map walks.
SplitPlan skewed3_plan(int64_t U, int sms) {
  SplitPlan pl = uniform_plan(3, U);
  pl.den = 4;
  pl.num[1] = 2; pl.num[2] = 3; pl.num[3] = 4;
  const int64_t x = 3 * U - sms;
  pl.push(0, x, 0, gdn::PrefillParams::kRunMaps);
  pl.push(0, x + U, 0, 0);
  pl.push(0, 3 * U, x, gdn::PrefillParams::kRunMaps);
  return pl;
}

// P = 4, segments of R, 1, 1, 2 parts of R + 4 (see the cost model above).
SplitPlan four_plan(int64_t U, int sms, int R) {
  SplitPlan pl = uniform_plan(4, U);
  pl.den = R + 4;
  pl.num[1] = R; pl.num[2] = R + 1; pl.num[3] = R + 2; pl.num[4] = R + 4;
  const int64_t m = sms - U, maps = 4 * U;
  // pass 1: CTA c < U walks segment 0 of (sequence, head) c; CTA U + i walks map walks
  // i, i + m, i + 2m, ... (indices c + r S of round r; the segment-0 CTAs are idle there)
  pl.push(0, U, 0, 0);
  int64_t u = U;
  for (int r = 0; r < R; ++r) {
    if (r > 0) {
      u = r * (int64_t)sms + U;
      pl.push(0, u, 0, gdn::PrefillParams::kRunIdle);
    }
    const int64_t cnt = std::min(m, maps - r * m);
    pl.push(0, u + cnt, r * m, gdn::PrefillParams::kRunMaps);
    u += cnt;
  }
  pl.units[0] = u;
  pl.grid[0] = (int)std::min<int64_t>(u, sms);
  // pass 2 (kinds 0, 1, 2 = segments 1, 2, 3) on 2U CTAs: CTA c < U re-runs segments 1 and
  // 2 of (sequence, head) c, CTA U + c segment 3
  pl.push(1, U, 0, 0);
  pl.push(1, 2 * U, 0, 2);
  pl.push(1, 3 * U, 0, 1);
  pl.units[1] = 3 * U;
  pl.grid[1] = (int)(2 * U);
  return pl;
}

// Testing aids of this host thread (gdn_testing_force_splits, gdn_testing_wait_limit).
thread_local int t_force_splits = 0;         // 0: the planner decides
thread_local uint64_t t_wait_ns = 0;         // 0: the default bound
thread_local int t_hold_local_ready = 0;

SplitPlan choose_splits(int64_t N, int64_t H, int64_t T, int sms) {
  const int64_t U = N * H;
  SplitPlan pl;
  if (t_force_splits > 0) {
    pl = uniform_plan(t_force_splits, U);
  } else if (sms > 0 && N > 0) {
    const int64_t chunks = (T / N + 63) / 64;
    double best = 0.8;
    for (int c = 2; c <= kMaxSplits && chunks >= 8 * c; ++c) {
      const int64_t w1 = (U * (2 * c - 3) + sms - 1) / sms, w2 = (U * (c - 1) + sms - 1) / sms;
      const double cost = double(w1 + w2) / c;
      if (cost < best) { best = cost; pl = uniform_plan(c, U); }
    }
    const int64_t extra = 3 * U - sms;
    if (extra > 0 && extra <= U && chunks >= 32) {
      const double cost = 0.5 + 0.25 * double((2 * U + sms - 1) / sms);
      if (cost < best) { best = cost; pl = skewed3_plan(U, sms); }
    }
    if (U < sms && 2 * U <= sms) {
      const int64_t m = sms - U;
      const int R = (int)((4 * U + m - 1) / m);
      if (R <= 3 && chunks >= 8 * (R + 4)) {
        const double cost = double(R + 2) / double(R + 4);
        if (cost < best) { best = cost; pl = four_plan(U, sms, R); }
      }
    }
  }
  while (pl.P > 1 && size_t(U) * size_t(gdn::split_ws_blocks(pl.P)) * 65536 > kMaxSplitWorkspace)
    pl = uniform_plan(pl.P - 1, U);
  return pl;
}

gdn_status_t ensure_workspace(DeviceState& d, size_t bytes, cudaStream_t stream) {
  if (bytes <= d.ws_bytes) return GDN_OK;
  // An allocation made while the stream is being captured would belong to the graph
  // (valid only while it runs), not to this library: the caller has to reserve first.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t ce = cudaStreamIsCapturing(stream, &cap);
  if (ce != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaStreamIsCapturing: %s", cudaGetErrorString(ce));
  if (cap != cudaStreamCaptureStatusNone)
    return fail(GDN_ERR_UNSUPPORTED,
                "split-K needs %zu B of workspace but %zu B are reserved and the stream is being "
                "captured: call gdn_reserve_workspace before the capture",
                bytes, d.ws_bytes);
  if (d.ws) {
    cudaError_t e = cudaFreeAsync(d.ws, stream);
    d.ws = nullptr;
    d.ws_bytes = 0;
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "split-K workspace release: %s", cudaGetErrorString(e));
  }
  void* ptr = nullptr;
  cudaError_t e = cudaMallocAsync(&ptr, bytes, stream);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "split-K workspace (%zu B): %s", bytes, cudaGetErrorString(e));
  d.ws = static_cast<float*>(ptr);
  d.ws_bytes = bytes;
  return GDN_OK;
}

// Set-up of the allocation-free entry point on the current device: the device
// checks, the tensor-map encoder and the address of the static scratch, once.
struct NoAllocState {
  bool ready = false;
  uint8_t* scratch = nullptr;  // kNoAllocHeaderBytes header, then the split-K workspace
};
NoAllocState g_na[kMaxDevices];

gdn_status_t noalloc_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (*dev < 0 || *dev >= kMaxDevices) return fail(GDN_ERR_INVALID_ARGUMENT, "device %d out of range", *dev);
  std::lock_guard<std::mutex> lk(g_mu);
  NoAllocState& d = g_na[*dev];
  if (d.ready) return GDN_OK;
  gdn_status_t st = check_device(*dev);
  if (st != GDN_OK) return st;
  if ((st = ensure_encode()) != GDN_OK) return st;
  void* base = nullptr;
  e = gdn::noalloc_scratch(&base);
  if (e != cudaSuccess || !base)
    return fail(GDN_ERR_CUDA, "static scratch address (cudaGetSymbolAddress): %s", cudaGetErrorString(e));
  d.scratch = static_cast<uint8_t*>(base);
  d.ready = true;
  return GDN_OK;
}

gdn_status_t current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  return init_device(*dev);
}

// Both prefill entry points.  `noalloc` selects the static scratch (and
// `device_error`, or the scratch's discard word) instead of the per-device
// allocations.
gdn_status_t chunk_prefill(const gdn_tensor_t* q, const gdn_tensor_t* k, const gdn_tensor_t* v,
                           const gdn_tensor_t* g, const gdn_tensor_t* beta, float scale,
                           const gdn_tensor_t* initial_state, const gdn_tensor_t* state_indices,
                           const gdn_tensor_t* output_state, const gdn_tensor_t* cu_seqlens, int use_qk_l2norm,
                           int batch_invariant, const gdn_tensor_t* output, cudaStream_t stream, bool noalloc,
                           int32_t* device_error, const gdn_tensor_t* checkpoints = nullptr,
                           int checkpoints_per_seq = 0, int checkpoint_every = 0) {
  gdn_status_t st;
  if ((st = check_qkv(q, "q")) != GDN_OK) return st;
  if ((st = check_qkv(k, "k")) != GDN_OK) return st;
  if ((st = check_qkv(v, "v")) != GDN_OK) return st;
  if (k->dtype != q->dtype || v->dtype != q->dtype) return fail(GDN_ERR_UNSUPPORTED, "q, k and v must share a dtype");
  if (k->shape[0] != q->shape[0] || k->shape[1] != q->shape[1])
    return fail(GDN_ERR_UNSUPPORTED, "q and k must have the same shape (H_q == H_k)");
  if (v->shape[0] != q->shape[0]) return fail(GDN_ERR_INVALID_ARGUMENT, "v has a different token count than q");
  const int64_t T = q->shape[0], Hqk = q->shape[1], Hv = v->shape[1];
  const int64_t H = Hqk > Hv ? Hqk : Hv;
  if (H % Hqk || H % Hv)
    return fail(GDN_ERR_UNSUPPORTED, "num_sab_heads %lld must be a multiple of H_qk %lld and H_v %lld", (long long)H,
                (long long)Hqk, (long long)Hv);
  if (H > (1 << 20)) return fail(GDN_ERR_UNSUPPORTED, "too many heads");
  if ((st = check_gate(g, "g", T, H, true)) != GDN_OK) return st;
  if ((st = check_gate(beta, "beta", T, H, true)) != GDN_OK) return st;
  if ((st = check_state(initial_state, "initial_state", H)) != GDN_OK) return st;
  if ((st = check_state(output_state, "output_state", H)) != GDN_OK) return st;
  if ((st = check_index_vec(cu_seqlens, "cu_seqlens", -1)) != GDN_OK) return st;
  const int64_t N = cu_seqlens->shape[0] - 1;
  if (N < 0) return fail(GDN_ERR_INVALID_ARGUMENT, "cu_seqlens needs at least one entry");
  if (N * H >= (int64_t(1) << 31)) return fail(GDN_ERR_UNSUPPORTED, "too many (sequence, head) units");
  if (state_indices && (st = check_index_vec(state_indices, "state_indices", N)) != GDN_OK) return st;
  if (!state_indices) {
    if (initial_state && initial_state->shape[0] < N)
      return fail(GDN_ERR_INVALID_ARGUMENT, "initial_state has %lld slots for %lld sequences",
                  (long long)initial_state->shape[0], (long long)N);
    if (output_state && output_state->shape[0] < N)
      return fail(GDN_ERR_INVALID_ARGUMENT, "output_state has %lld slots for %lld sequences",
                  (long long)output_state->shape[0], (long long)N);
  }
  if ((st = check_basic(output, "output", 3)) != GDN_OK) return st;
  if (output->dtype != q->dtype) return fail(GDN_ERR_UNSUPPORTED, "output must have q's dtype");
  if (output->shape[0] != T || output->shape[1] != H || output->shape[2] != 128)
    return fail(GDN_ERR_INVALID_ARGUMENT, "output must be [T=%lld, H=%lld, 128]", (long long)T, (long long)H);
  if (output->stride[2] != 1 || (T > 0 && ((output->stride[0] % 8) || (output->stride[1] % 8) ||
                                           reinterpret_cast<uintptr_t>(output->data) % 16)))
    return fail(GDN_ERR_INVALID_ARGUMENT, "output rows must be contiguous and 16-byte aligned");
  if (!std::isfinite(scale)) return fail(GDN_ERR_INVALID_ARGUMENT, "scale must be finite");
  const float sc = (scale == 0.0f) ? 1.0f / std::sqrt(128.0f) : scale;

  if (overlaps(output_state, initial_state))
    return fail(GDN_ERR_ALIAS, "output_state must not overlap initial_state");
  const gdn_tensor_t* ins[] = {q, k, v, g, beta, initial_state, cu_seqlens, state_indices};
  for (const gdn_tensor_t* in : ins) {
    if (overlaps(output, in)) return fail(GDN_ERR_ALIAS, "output overlaps an input");
    if (overlaps(output_state, in)) return fail(GDN_ERR_ALIAS, "output_state overlaps an input");
  }
  if (overlaps(output, output_state)) return fail(GDN_ERR_ALIAS, "output overlaps output_state");
  if (checkpoints) {
    if ((st = check_basic(checkpoints, "checkpoints", 4)) != GDN_OK) return st;
    if (checkpoints->dtype != GDN_F32) return fail(GDN_ERR_UNSUPPORTED, "checkpoints must be f32");
    if (checkpoints_per_seq < 1) return fail(GDN_ERR_INVALID_ARGUMENT, "checkpoints_per_seq must be >= 1");
    if (checkpoints->shape[0] != N * checkpoints_per_seq || checkpoints->shape[1] != H ||
        checkpoints->shape[2] != 128 || checkpoints->shape[3] != 128)
      return fail(GDN_ERR_INVALID_ARGUMENT, "checkpoints must be [N * M = %lld, H=%lld, 128, 128]",
                  (long long)(N * checkpoints_per_seq), (long long)H);
    if (checkpoints->stride[3] != 1 || checkpoints->stride[2] != 128 || (checkpoints->stride[0] % 4) ||
        (checkpoints->stride[1] % 4) || reinterpret_cast<uintptr_t>(checkpoints->data) % 16)
      return fail(GDN_ERR_INVALID_ARGUMENT, "checkpoint blocks must be contiguous 128 x 128 with 16-byte aligned rows");
    if (checkpoint_every < 1) return fail(GDN_ERR_INVALID_ARGUMENT, "checkpoint_every must be >= 1 chunk");
    const gdn_tensor_t* all[] = {q, k, v, g, beta, initial_state, cu_seqlens, state_indices, output, output_state};
    for (const gdn_tensor_t* x : all)
      if (overlaps(checkpoints, x)) return fail(GDN_ERR_ALIAS, "checkpoints overlap another argument");
  }

  int dev = 0;
  if ((st = noalloc ? noalloc_device(&dev) : current_device(&dev)) != GDN_OK) return st;
  if (N == 0) return GDN_OK;

  gdn::PrefillParams p;
  memset(&p, 0, sizeof(p));
  if ((st = encode_qkv(&p.tm_q, q, "q")) != GDN_OK) return st;
  if ((st = encode_qkv(&p.tm_k, k, "k")) != GDN_OK) return st;
  if ((st = encode_qkv(&p.tm_v, v, "v")) != GDN_OK) return st;
  if ((st = encode_out(&p.tm_o, output)) != GDN_OK) return st;
  if (g) { p.g = g->data; p.g_st = g->stride[0]; p.g_sh = g->stride[1]; p.g_dtype = g->dtype; }
  if (beta) { p.beta = beta->data; p.b_st = beta->stride[0]; p.b_sh = beta->stride[1]; p.b_dtype = beta->dtype; }
  if (initial_state) {
    p.s_in = initial_state->data; p.sin_slot = initial_state->stride[0]; p.sin_head = initial_state->stride[1];
    p.sin_slots = initial_state->shape[0]; p.sin_dtype = initial_state->dtype;
    p.sin_tma = encode_state_pool(&p.tm_sin, initial_state) ? 1 : 0;
  }
  if (output_state) {
    p.s_out = output_state->data; p.sout_slot = output_state->stride[0]; p.sout_head = output_state->stride[1];
    p.sout_slots = output_state->shape[0]; p.sout_dtype = output_state->dtype;
    p.sout_tma = encode_state_pool(&p.tm_sout, output_state) ? 1 : 0;
  }
  if (state_indices) { p.state_idx = state_indices->data; p.idx_dtype = state_indices->dtype; }
  p.cu = cu_seqlens->data;
  p.cu_dtype = cu_seqlens->dtype;
  p.out = output->data;
  p.o_st = output->stride[0];
  p.o_sh = output->stride[1];
  if (noalloc) {
    int32_t* discard = reinterpret_cast<int32_t*>(g_na[dev].scratch);
    if (!device_error) {
      cudaError_t e = cudaMemsetAsync(discard, 0, sizeof(int32_t), stream);
      if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "clearing the scratch error word: %s", cudaGetErrorString(e));
    }
    p.dev_err = device_error ? device_error : discard;
  } else {
    p.dev_err = g_dev[dev].dev_err;
  }
  p.T = T;
  p.N = (int32_t)N;
  p.H = (int32_t)H;
  p.H_qk = (int32_t)Hqk;
  p.H_v = (int32_t)Hv;
  p.scale = sc;
  p.l2norm = use_qk_l2norm ? 1 : 0;
  p.op_f16 = q->dtype == GDN_F16 ? 1 : 0;
  p.wait_ns = t_wait_ns ? t_wait_ns : 200ull * 1000 * 1000;
  p.hold_local_ready = t_hold_local_ready;
  if (checkpoints) {
    p.ck = static_cast<float*>(checkpoints->data);
    p.ck_seq = checkpoints->stride[0] * checkpoints_per_seq;
    p.ck_idx = checkpoints->stride[0];
    p.ck_head = checkpoints->stride[1];
    p.ck_count = checkpoints_per_seq;
    p.ck_every = checkpoint_every;
  }
  const SplitPlan plan = batch_invariant ? SplitPlan() : choose_splits(N, H, T, gdn::device_sm_count());
  const int P = plan.P;
  if (P == 1) {  // one CTA walks each (sequence, head) from its first chunk to its last
    p.mode = 0;
    p.splits = 1;
    p.n_units = N * H;
    cudaError_t e = gdn::launch_prefill(p, stream);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    return GDN_OK;
  }
  // split-K: pass 1 (segment 0 + middle-segment maps), fix-up, pass 2 (segments 1..P-1)
  const size_t ws_bytes = size_t(N * H) * size_t(gdn::split_ws_blocks(P)) * 65536;
  if (noalloc) {
    if (ws_bytes > gdn::kNoAllocWorkspaceBytes)
      return fail(GDN_ERR_UNSUPPORTED,
                  "split-K with P = %d needs %zu B of workspace; the static scratch holds %zu B (pass "
                  "batch_invariant = 1, or use gdn_chunk_prefill)",
                  P, ws_bytes, gdn::kNoAllocWorkspaceBytes);
    p.ws = reinterpret_cast<float*>(g_na[dev].scratch + gdn::kNoAllocHeaderBytes);
  } else {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = ensure_workspace(g_dev[dev], ws_bytes, stream)) != GDN_OK) return st;
    p.ws = g_dev[dev].ws;
  }
  p.splits = P;
  for (int i = 0; i <= P; ++i) p.seg_num[i] = plan.num[i];
  p.seg_den = plan.den;
  cudaError_t e = cudaSuccess;
  for (int pass = 0; pass < 2 && e == cudaSuccess; ++pass) {
    p.mode = pass + 1;
    p.n_units = plan.units[pass];
    p.grid = plan.grid[pass];
    p.n_runs = plan.n_runs[pass];
    for (int r = 0; r < plan.n_runs[pass]; ++r) p.runs[r] = plan.runs[pass][r];
    e = gdn::launch_prefill(p, stream);
    if (e == cudaSuccess && pass == 0) e = gdn::launch_split_fixup(p, stream);
  }
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "split-K prefill launch (P = %d): %s", P, cudaGetErrorString(e));
  return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status_t gdn_init(int device) {
  g_last_error[0] = 0;
  return init_device(device);
}

const char* gdn_last_error(void) { return g_last_error; }

gdn_status_t gdn_chunk_prefill(const gdn_tensor_t* q, const gdn_tensor_t* k, const gdn_tensor_t* v,
                               const gdn_tensor_t* g, const gdn_tensor_t* beta, float scale,
                               const gdn_tensor_t* initial_state, const gdn_tensor_t* state_indices,
                               const gdn_tensor_t* output_state, const gdn_tensor_t* cu_seqlens,
                               int use_qk_l2norm, int batch_invariant, const gdn_tensor_t* output,
                               cudaStream_t stream) {
  g_last_error[0] = 0;
  return chunk_prefill(q, k, v, g, beta, scale, initial_state, state_indices, output_state, cu_seqlens,
                       use_qk_l2norm, batch_invariant, output, stream, false, nullptr);
}

gdn_status_t gdn_chunk_prefill_checkpointed(const gdn_tensor_t* q, const gdn_tensor_t* k, const gdn_tensor_t* v,
                                            const gdn_tensor_t* g, const gdn_tensor_t* beta, float scale,
                                            const gdn_tensor_t* initial_state, const gdn_tensor_t* state_indices,
                                            const gdn_tensor_t* output_state, const gdn_tensor_t* cu_seqlens,
                                            int use_qk_l2norm, int batch_invariant, const gdn_tensor_t* output,
                                            const gdn_tensor_t* checkpoints, int checkpoints_per_seq,
                                            int checkpoint_every, cudaStream_t stream) {
  g_last_error[0] = 0;
  if (!checkpoints) return fail(GDN_ERR_INVALID_ARGUMENT, "checkpoints is required");
  return chunk_prefill(q, k, v, g, beta, scale, initial_state, state_indices, output_state, cu_seqlens,
                       use_qk_l2norm, batch_invariant, output, stream, false, nullptr, checkpoints,
                       checkpoints_per_seq, checkpoint_every);
}

gdn_status_t gdn_chunk_prefill_noalloc(const gdn_tensor_t* q, const gdn_tensor_t* k, const gdn_tensor_t* v,
                                       const gdn_tensor_t* g, const gdn_tensor_t* beta, float scale,
                                       const gdn_tensor_t* initial_state, const gdn_tensor_t* state_indices,
                                       const gdn_tensor_t* output_state, const gdn_tensor_t* cu_seqlens,
                                       int use_qk_l2norm, int batch_invariant, const gdn_tensor_t* output,
                                       int32_t* device_error, cudaStream_t stream) {
  g_last_error[0] = 0;
  return chunk_prefill(q, k, v, g, beta, scale, initial_state, state_indices, output_state, cu_seqlens,
                       use_qk_l2norm, batch_invariant, output, stream, true, device_error);
}

gdn_status_t gdn_decode_step(const gdn_tensor_t* q, const gdn_tensor_t* k, const gdn_tensor_t* v,
                             const gdn_tensor_t* g, const gdn_tensor_t* beta, float scale,
                             const gdn_tensor_t* state, const gdn_tensor_t* state_indices, int use_qk_l2norm,
                             const gdn_tensor_t* output, cudaStream_t stream) {
  g_last_error[0] = 0;
  gdn_status_t st;
  if ((st = check_qkv(q, "q")) != GDN_OK) return st;
  if ((st = check_qkv(k, "k")) != GDN_OK) return st;
  if ((st = check_qkv(v, "v")) != GDN_OK) return st;
  if (k->dtype != q->dtype || v->dtype != q->dtype) return fail(GDN_ERR_UNSUPPORTED, "q, k and v must share a dtype");
  if (k->shape[0] != q->shape[0] || k->shape[1] != q->shape[1])
    return fail(GDN_ERR_UNSUPPORTED, "q and k must have the same shape (H_q == H_k)");
  if (v->shape[0] != q->shape[0]) return fail(GDN_ERR_INVALID_ARGUMENT, "v has a different batch size than q");
  const int64_t B = q->shape[0], Hqk = q->shape[1], Hv = v->shape[1];
  const int64_t H = Hqk > Hv ? Hqk : Hv;
  if (H % Hqk || H % Hv)
    return fail(GDN_ERR_UNSUPPORTED, "num_sab_heads %lld must be a multiple of H_qk %lld and H_v %lld", (long long)H,
                (long long)Hqk, (long long)Hv);
  if (B * H >= (int64_t(1) << 28)) return fail(GDN_ERR_UNSUPPORTED, "too many (row, head) states");
  if ((st = check_gate(g, "g", B, H, true)) != GDN_OK) return st;
  if ((st = check_gate(beta, "beta", B, H, true)) != GDN_OK) return st;
  if (!state) return fail(GDN_ERR_INVALID_ARGUMENT, "state is required");
  if ((st = check_state(state, "state", H)) != GDN_OK) return st;
  if (state_indices && (st = check_index_vec(state_indices, "state_indices", B)) != GDN_OK) return st;
  if (!state_indices && state->shape[0] < B)
    return fail(GDN_ERR_INVALID_ARGUMENT, "state has %lld slots for %lld rows", (long long)state->shape[0],
                (long long)B);
  if ((st = check_basic(output, "output", 3)) != GDN_OK) return st;
  if (output->dtype != q->dtype) return fail(GDN_ERR_UNSUPPORTED, "output must have q's dtype");
  if (output->shape[0] != B || output->shape[1] != H || output->shape[2] != 128 || output->stride[2] != 1)
    return fail(GDN_ERR_INVALID_ARGUMENT, "output must be [B=%lld, H=%lld, 128] with contiguous rows", (long long)B,
                (long long)H);
  if (!std::isfinite(scale)) return fail(GDN_ERR_INVALID_ARGUMENT, "scale must be finite");
  const gdn_tensor_t* ins[] = {q, k, v, g, beta, state_indices};
  for (const gdn_tensor_t* in : ins) {
    if (overlaps(output, in)) return fail(GDN_ERR_ALIAS, "output overlaps an input");
    if (overlaps(state, in)) return fail(GDN_ERR_ALIAS, "state overlaps an input");
  }
  if (overlaps(output, state)) return fail(GDN_ERR_ALIAS, "output overlaps state");
  int dev = 0;
  if ((st = current_device(&dev)) != GDN_OK) return st;
  if (B == 0) return GDN_OK;
  gdn::DecodeParams p;
  memset(&p, 0, sizeof(p));
  p.q = q->data; p.q_sb = q->stride[0]; p.q_sh = q->stride[1];
  p.k = k->data; p.k_sb = k->stride[0]; p.k_sh = k->stride[1];
  p.v = v->data; p.v_sb = v->stride[0]; p.v_sh = v->stride[1];
  if (g) { p.g = g->data; p.g_sb = g->stride[0]; p.g_sh = g->stride[1]; p.g_dtype = g->dtype; }
  if (beta) { p.beta = beta->data; p.b_sb = beta->stride[0]; p.b_sh = beta->stride[1]; p.b_dtype = beta->dtype; }
  p.state = state->data; p.st_slot = state->stride[0]; p.st_head = state->stride[1];
  p.st_slots = state->shape[0]; p.st_dtype = state->dtype;
  if (state_indices) { p.state_idx = state_indices->data; p.idx_dtype = state_indices->dtype; }
  p.out = output->data; p.o_sb = output->stride[0]; p.o_sh = output->stride[1];
  p.dev_err = g_dev[dev].dev_err;
  p.B = (int32_t)B; p.H = (int32_t)H; p.H_qk = (int32_t)Hqk; p.H_v = (int32_t)Hv;
  p.scale = (scale == 0.0f) ? 1.0f / std::sqrt(128.0f) : scale;
  p.l2norm = use_qk_l2norm ? 1 : 0;
  p.in_f16 = q->dtype == GDN_F16 ? 1 : 0;
  cudaError_t e = gdn::launch_decode(p, stream);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return GDN_OK;
}

gdn_status_t gdn_reserve_workspace(size_t bytes, cudaStream_t stream) {
  g_last_error[0] = 0;
  int dev = 0;
  gdn_status_t st = current_device(&dev);
  if (st != GDN_OK) return st;
  std::lock_guard<std::mutex> lk(g_mu);
  return ensure_workspace(g_dev[dev], bytes, stream);
}

size_t gdn_split_workspace_bytes(int64_t num_seqs, int64_t num_sab_heads, int splits) {
  if (num_seqs <= 0 || num_sab_heads <= 0 || splits < 2) return 0;
  return size_t(num_seqs) * size_t(num_sab_heads) * size_t(gdn::split_ws_blocks(splits)) * 65536;
}

gdn_status_t gdn_get_device_status(cudaStream_t stream, int32_t* device_error) {
  g_last_error[0] = 0;
  if (!device_error) return fail(GDN_ERR_INVALID_ARGUMENT, "device_error is null");
  *device_error = 0;
  int dev = 0;
  gdn_status_t st = current_device(&dev);
  if (st != GDN_OK) return st;
  cudaError_t e = cudaStreamSynchronize(stream);
  int32_t word = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&word, g_dev[dev].dev_err, sizeof(word), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(g_dev[dev].dev_err, 0, sizeof(word));
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "reading the device error word: %s", cudaGetErrorString(e));
  *device_error = word;
  if (word) return fail(GDN_ERR_DEVICE_INPUT, "device-detected input error bits 0x%x", word);
  return GDN_OK;
}

gdn_status_t gdn_testing_force_splits(int splits) {
  g_last_error[0] = 0;
  if (splits < 0 || splits > kMaxSplits) return fail(GDN_ERR_INVALID_ARGUMENT, "splits must be 0..%d", kMaxSplits);
  t_force_splits = splits;
  return GDN_OK;
}

gdn_status_t gdn_testing_wait_limit(uint64_t limit_ns, int withhold_local_ready) {
  g_last_error[0] = 0;
  if (limit_ns != 0 && limit_ns < 1000)
    return fail(GDN_ERR_INVALID_ARGUMENT, "a wait limit below 1 us is not supported");
  t_wait_ns = limit_ns;
  t_hold_local_ready = withhold_local_ready ? 1 : 0;
  return GDN_OK;
}

gdn_status_t gdn_testing_split_plan(int64_t num_seqs, int64_t num_heads, int64_t total_tokens, int num_sms,
                                    int32_t* plan, int32_t* units, int64_t capacity) {
  g_last_error[0] = 0;
  if (num_seqs <= 0 || num_heads <= 0 || total_tokens < 0 || num_sms <= 0 || !plan)
    return fail(GDN_ERR_INVALID_ARGUMENT, "split plan: sizes must be positive and plan non-null");
  const SplitPlan pl = choose_splits(num_seqs, num_heads, total_tokens, num_sms);
  for (int i = 0; i < 16; ++i) plan[i] = 0;
  plan[0] = pl.P;
  plan[1] = pl.den;
  for (int i = 0; i <= pl.P; ++i) plan[2 + i] = pl.num[i];
  if (pl.P == 1) return GDN_OK;
  gdn::PrefillParams p;
  memset(&p, 0, sizeof(p));
  p.splits = pl.P;
  for (int pass = 0; pass < 2; ++pass) {
    const int64_t n = pl.units[pass];
    plan[11 + pass] = pl.grid[pass] > 0 ? pl.grid[pass] : (int32_t)std::min<int64_t>(n, num_sms);
    plan[13 + pass] = (int32_t)n;
    if (!units || capacity < n) return fail(GDN_ERR_INVALID_ARGUMENT, "split plan: capacity %lld below %lld units",
                                            (long long)capacity, (long long)n);
    p.mode = pass + 1;
    p.n_runs = pl.n_runs[pass];
    for (int r = 0; r < pl.n_runs[pass]; ++r) p.runs[r] = pl.runs[pass][r];
    int32_t* out = units + (int64_t)pass * capacity * 2;
    for (int64_t u = 0; u < n; ++u) {
      int32_t nh = -1, kind = -1;
      if (!gdn::split_unit(p, u, &nh, &kind)) nh = kind = -1;
      out[2 * u] = nh;
      out[2 * u + 1] = kind;
    }
  }
  return GDN_OK;
}

void gdn_shutdown(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int prev = -1;
  cudaGetDevice(&prev);
  for (int d = 0; d < kMaxDevices; ++d) {
    if (g_dev[d].dev_err || g_dev[d].ws) {
      cudaSetDevice(d);
      if (g_dev[d].dev_err) cudaFree(g_dev[d].dev_err);
      if (g_dev[d].ws) cudaFree(g_dev[d].ws);
    }
    g_dev[d] = DeviceState();
    g_na[d] = NoAllocState();  // the static scratch's address is looked up again (it lives as long as the context)
  }
  gdn::invalidate_launch_config();  // kernel attributes are set again on every thread's next launch
  if (prev >= 0) cudaSetDevice(prev);
}

}  // extern "C"
