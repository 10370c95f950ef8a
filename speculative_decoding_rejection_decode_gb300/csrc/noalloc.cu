// Allocation-free entry point: specdec_rejection_sample_noalloc.
//
// Some callers cannot call cudaMalloc at the point where they verify: code that
// runs inside a memory pool or arena they do not own, plug-ins that are given
// only pre-allocated buffers, or hosts that forbid device allocation after
// start-up so that memory use stays fixed.  For them this entry point runs the
// same kernels as specdec_rejection_sample, but its scratch (per-row softmax
// statistics and status words, the deferred-request list and a few counters)
// lives in one file-scope __device__ array of fixed size instead of a
// handle-owned allocation.  Every GPU that loads the library holds that array
// until the process exits.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "kernels.cuh"

using namespace specdec;

namespace {

constexpr int64_t kRows = SPECDEC_NOALLOC_MAX_ROWS;
constexpr int kBatch = SPECDEC_NOALLOC_MAX_BATCH;
constexpr int kThreads = 512;  // sweep kernel: 2 CTAs of 512 threads per SM
constexpr int kSlices = 16;    // race slices per deferred request (keeps the scratch small)

constexpr size_t kStatsOff = 0;
constexpr size_t kStatusOff = kStatsOff + kRows * sizeof(float2);
constexpr size_t kKeysOff = kStatusOff + kRows * sizeof(uint64_t);
constexpr size_t kNaccOff = kKeysOff + kRows * sizeof(uint64_t);
constexpr size_t kListOff = kNaccOff + kBatch * sizeof(int32_t);
constexpr size_t kRpartOff = kListOff + kBatch * sizeof(int32_t);
constexpr size_t kRcountOff = kRpartOff + (size_t)kBatch * kSlices * sizeof(float4);
constexpr size_t kSmallOff = kRcountOff + kBatch * sizeof(int32_t);  // err, defer count, counter
constexpr size_t kSmallBytes = 64;
constexpr size_t kScratchBytes = kSmallOff + kSmallBytes;
static_assert(kStatusOff % 256 == 0 && kKeysOff % 256 == 0 && kNaccOff % 256 == 0 &&
                  kListOff % 256 == 0 && kRpartOff % 256 == 0 && kRcountOff % 256 == 0 &&
                  kSmallOff % 256 == 0,
              "scratch sections stay 256-byte aligned");

}  // namespace

// The scratch array.  In host code this name is only a stand-in: its device
// address comes from cudaGetSymbolAddress (below).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
std::atomic<uint64_t> g_epoch{0};

// Device address of the scratch array on the current device.  It is looked up
// on every call made outside stream capture (a host-side query), so that a
// module loaded again after cudaDeviceReset is found at its new address; a
// call made while `st` is capturing uses the address of the last call on this
// device outside capture (a lookup may not be legal there), so the first call
// on a device has to come before any capture.
int scratch_on_current_device(cudaStream_t st, unsigned char** out, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPECDEC_ERR_CUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SPECDEC_ERR_CUDA;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return SPECDEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return SPECDEC_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  } else if (!g_scratch_ptr[dev]) {
    return SPECDEC_ERR_CUDA;
  }
  *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
  return SPECDEC_OK;
}

}  // namespace

extern "C" int specdec_rejection_sample_noalloc(
    const void* target_logits, int dtype, const float* draft_probs, const int32_t* draft_ids,
    const int32_t* cu_num_draft_tokens, int B, int V, float T, uint64_t seed,
    int64_t n_draft_positions, int32_t* out_tokens, int32_t* out_num_accepted, float* out_beta,
    uint32_t* out_device_error, void* stream) {
  if (dtype != SPECDEC_F32 && dtype != SPECDEC_BF16) return SPECDEC_ERR_UNSUPPORTED_DTYPE;
  if (B <= 0 || V <= 0 || V > (1 << 30) || n_draft_positions < 0) return SPECDEC_ERR_INVALID_ARG;
  if (!std::isfinite(T) || T < 0.0f) return SPECDEC_ERR_INVALID_ARG;
  if (!target_logits || !draft_ids || !cu_num_draft_tokens || !out_tokens || !out_num_accepted)
    return SPECDEC_ERR_INVALID_ARG;
  if (B > kBatch || n_draft_positions + B > kRows) return SPECDEC_ERR_CAPACITY;

  unsigned char* base = nullptr;
  int sms = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = scratch_on_current_device(st, &base, &sms);
  if (rc != SPECDEC_OK) return rc;
  uint32_t* small = reinterpret_cast<uint32_t*>(base + kSmallOff);
  // Everything a call accumulates into starts at zero on its stream: the small
  // block (error word, deferred count, work counter), the greedy argmax keys
  // (T == 0) and the per-request slice counters of the race (T > 0).  A call
  // that completes leaves the keys and the slice counters at zero itself; these
  // clears also cover an earlier call that stopped part-way.  Status words need
  // no clearing (each call tags them with its own epoch).
  if (cudaMemsetAsync(small, 0, kSmallBytes, st) != cudaSuccess) return SPECDEC_ERR_CUDA;
  if (T == 0.0f) {
    if (cudaMemsetAsync(base + kKeysOff, 0, kRows * sizeof(uint64_t), st) != cudaSuccess)
      return SPECDEC_ERR_CUDA;
  } else if (cudaMemsetAsync(base + kRcountOff, 0, kBatch * sizeof(int32_t), st) != cudaSuccess) {
    return SPECDEC_ERR_CUDA;
  }

  Params P = {};
  P.logits = target_logits;
  P.q = draft_probs;
  P.ids = draft_ids;
  P.cu = cu_num_draft_tokens;
  P.B = B;
  P.V = V;
  P.c = T > 0.0f ? kLog2e / T : 0.0f;
  P.seed = seed;
  P.req_offset = 0;
  P.epoch = ++g_epoch;
  P.out_tokens = out_tokens;
  P.out_nacc = out_num_accepted;
  P.out_beta = out_beta;
  P.row_stats = reinterpret_cast<float2*>(base + kStatsOff);
  P.status = reinterpret_cast<uint64_t*>(base + kStatusOff);
  P.gkeys = reinterpret_cast<uint64_t*>(base + kKeysOff);
  P.ws_nacc = reinterpret_cast<int32_t*>(base + kNaccOff);
  P.defer_list = reinterpret_cast<int32_t*>(base + kListOff);
  P.rpart = reinterpret_cast<float4*>(base + kRpartOff);
  P.rcount = reinterpret_cast<int32_t*>(base + kRcountOff);
  P.rslices = (int)std::min<int64_t>(kSlices, std::max<int64_t>(1, (V + 4095) / 4096));
  P.rslice_len = (int)(((V + P.rslices - 1) / P.rslices + 7) / 8 * 8);
  P.rstride = kSlices;
  P.err = out_device_error ? out_device_error : small;
  P.defer_count = reinterpret_cast<int32_t*>(small + 1);
  P.sched = reinterpret_cast<unsigned long long*>(small + 2);
  P.cap_rows = kRows;
  P.cap_b = kBatch;

  const int esize = dtype == SPECDEC_BF16 ? 2 : 4;
  if (T == 0.0f) {
    const int vec_ok = ((int64_t)V * esize) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(target_logits) % 16 == 0;
    if (dtype == SPECDEC_BF16)
      greedy_partial_kernel<__nv_bfloat16><<<sms * 8, kRowThreads, 0, st>>>(P, vec_ok);
    else
      greedy_partial_kernel<float><<<sms * 8, kRowThreads, 0, st>>>(P, vec_ok);
    if (launch_dependent(greedy_finalize_kernel, (B + 7) / 8, 256, st, P) != cudaSuccess)
      return SPECDEC_ERR_CUDA;
  } else {
    P.vec_ok = ((int64_t)V * esize) % 16 == 0 && ((int64_t)V * 4) % 16 == 0 &&
               reinterpret_cast<uintptr_t>(target_logits) % 16 == 0 &&
               reinterpret_cast<uintptr_t>(draft_probs) % 16 == 0;
    const int race_grid = sms * 8;
    cudaError_t e;
    // one-hot drafts: eight 128-thread CTAs per SM (racing CTAs and streaming
    // ones share each SM), as on the handle path
    const bool onehot = draft_probs == nullptr;
    if (dtype == SPECDEC_BF16) {
      if (onehot)
        sweep_row_kernel<__nv_bfloat16, 128, 8><<<sms * 8, 128, 0, st>>>(P);
      else
        sweep_row_kernel<__nv_bfloat16, kThreads, 2><<<sms * 2, kThreads, 0, st>>>(P);
      e = launch_dependent(finalize_kernel, (B + 255) / 256, 256, st, P);
      if (e == cudaSuccess) e = launch_dependent(race_kernel<__nv_bfloat16>, race_grid, kRowThreads, st, P);
    } else {
      if (onehot)
        sweep_row_kernel<float, 128, 8><<<sms * 8, 128, 0, st>>>(P);
      else
        sweep_row_kernel<float, kThreads, 2><<<sms * 2, kThreads, 0, st>>>(P);
      e = launch_dependent(finalize_kernel, (B + 255) / 256, 256, st, P);
      if (e == cudaSuccess) e = launch_dependent(race_kernel<float>, race_grid, kRowThreads, st, P);
    }
    if (e != cudaSuccess) return SPECDEC_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}
