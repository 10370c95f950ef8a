// Host side of libspecdec.so: argument checks, workspace, path choice and
// launches.  The C ABI is declared (and documented) in include/specdec.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>

#include "kernels.cuh"
#include "tree.cuh"

using namespace specdec;

namespace {

constexpr int kClusterSizes[5] = {1, 2, 4, 8, 16};
constexpr int kMinRing = 3;  // draft ring stages the fused kernel needs at least

struct Workspace {
  void* base = nullptr;
  int64_t cap_rows = 0;
  int cap_b = 0;
  float2* row_stats = nullptr;
  float* row_tau = nullptr;
  uint64_t* status = nullptr;
  uint64_t* gkeys = nullptr;
  int32_t* ws_nacc = nullptr;
  int32_t* defer_list = nullptr;
  float4* rpart = nullptr;
  int32_t* rcount = nullptr;
  float4* dual_part = nullptr;
  int32_t* dual_cnt = nullptr;
  unsigned long long* dual_skip = nullptr;
  unsigned long long* dual_race = nullptr;
};

struct FusedConfig {
  bool ok = false;
  int C = 0, slice_len = 0, tbuf_bytes = 0, nq = 0, smem = 0, clusters = 0;
};

}  // namespace

struct specdec_ctx {
  int device = 0;
  int num_sms = 0;
  int smem_optin = 0;
  Workspace ws;
  uint32_t* small = nullptr;  // [0] sticky error word, [1] deferred-request count,
                              // [2..3] sweep-kernel work counter (64-bit),
                              // [4..5] tree-walk request counter (64-bit)
  bool reserved = false;
  int64_t res_rows = 0;
  int res_b = 0;
  uint64_t epoch = 0;
  int path_override = SPECDEC_PATH_AUTO;
  int last_path = 0, last_cluster = 0;
  cudaEvent_t ev_before = nullptr, ev_after = nullptr;
  int stream_smem[4] = {0, 0, 0, 0};  // dynamic shared memory set on stream_row_kernel<dtype, ctas>
  int smem_per_sm = 0;
  int sweep_threads = 0;        // block size of the sweep kernel (1024 x 1 .. 64 x 16 per SM; 0: by call)
  int sweep_ctas = 0;           // grid of the 512-thread sweep kernel (0: two per SM)
  int stream_ctas = 1;          // stream kernel CTAs per SM (1 or 2)
  int pair_clusters[2][2] = {{0, 0}, {0, 0}};  // co-resident 2-CTA clusters of pair_row_kernel<f32 / bf16, 512 / 256>
  int pair_threads = 512;           // pair kernel block size (512: 2 CTAs per SM, or 256: 4)
  int occ_cache[2][5][2] = {};  // [dtype][cluster index] -> {smem, clusters}
  int adj_smem_set[2][2] = {{0, 0}, {0, 0}};  // dynamic shared memory set on the adjusted sweep kernel
  int adj_threads = 512;            // adjusted sweep kernel block size (512: 2 CTAs per SM, or 1024: 1)
  unsigned long long* adj_ctr = nullptr;  // caller's selection counters (profiling), or null
  int fault_mode = 0;           // specdec_set_fault_injection
  uint64_t fault_wait_ns = 0;
};

namespace {

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Makes the handle's device current for one entry-point call and puts the
// caller's current device back when the call returns, so that no call changes
// which device the calling thread works on.
class DeviceGuard {
 public:
  explicit DeviceGuard(int device) {
    if (cudaGetDevice(&prev_) != cudaSuccess) {
      cudaGetLastError();
      prev_ = -1;
    }
    ok_ = prev_ == device || cudaSetDevice(device) == cudaSuccess;
    restore_ = ok_ && prev_ >= 0 && prev_ != device;
  }
  ~DeviceGuard() {
    if (restore_) cudaSetDevice(prev_);
  }
  DeviceGuard(const DeviceGuard&) = delete;
  DeviceGuard& operator=(const DeviceGuard&) = delete;
  bool ok() const { return ok_; }

 private:
  int prev_ = -1;
  bool ok_ = false;
  bool restore_ = false;
};

int free_workspace(specdec_ctx* h) {
  if (h->ws.base) {
    cudaFree(h->ws.base);
    h->ws = Workspace{};
  }
  return SPECDEC_OK;
}

int alloc_workspace(specdec_ctx* h, int64_t rows, int b) {
  rows = std::max<int64_t>(rows, 1);
  b = std::max(b, 1);
  const size_t stats_b = round_up(rows * sizeof(float2), 256);
  const size_t tau_b = round_up(rows * sizeof(float), 256);
  const size_t status_b = round_up(rows * sizeof(uint64_t), 256);
  const size_t gkeys_b = round_up(rows * sizeof(uint64_t), 256);
  const size_t nacc_b = round_up((size_t)b * sizeof(int32_t), 256);
  const size_t list_b = nacc_b;
  const size_t rpart_b = round_up((size_t)b * kRaceMaxSlices * sizeof(float4), 256);
  const size_t rcount_b = nacc_b;
  const size_t dpart_b = round_up(rows * 2 * sizeof(float4), 256);
  const size_t dcnt_b = round_up(rows * sizeof(int32_t), 256);
  const size_t ddec_b = round_up(rows * sizeof(unsigned long long), 256);
  const size_t total = stats_b + tau_b + status_b + gkeys_b + nacc_b + list_b + rpart_b + rcount_b +
                       dpart_b + dcnt_b + 2 * ddec_b;
  if (cudaDeviceSynchronize() != cudaSuccess) return SPECDEC_ERR_CUDA;
  free_workspace(h);
  void* p = nullptr;
  if (cudaMalloc(&p, total) != cudaSuccess) {
    cudaGetLastError();
    return SPECDEC_ERR_OOM;
  }
  if (cudaMemset(p, 0, total) != cudaSuccess) {
    cudaFree(p);
    return SPECDEC_ERR_CUDA;
  }
  char* c = static_cast<char*>(p);
  h->ws.base = p;
  h->ws.row_stats = reinterpret_cast<float2*>(c);
  c += stats_b;
  h->ws.row_tau = reinterpret_cast<float*>(c);
  c += tau_b;
  h->ws.status = reinterpret_cast<uint64_t*>(c);
  c += status_b;
  h->ws.gkeys = reinterpret_cast<uint64_t*>(c);
  c += gkeys_b;
  h->ws.ws_nacc = reinterpret_cast<int32_t*>(c);
  c += nacc_b;
  h->ws.defer_list = reinterpret_cast<int32_t*>(c);
  c += list_b;
  h->ws.rpart = reinterpret_cast<float4*>(c);
  c += rpart_b;
  h->ws.rcount = reinterpret_cast<int32_t*>(c);
  c += rcount_b;
  h->ws.dual_part = reinterpret_cast<float4*>(c);
  c += dpart_b;
  h->ws.dual_cnt = reinterpret_cast<int32_t*>(c);
  c += dcnt_b;
  h->ws.dual_skip = reinterpret_cast<unsigned long long*>(c);
  c += ddec_b;
  h->ws.dual_race = reinterpret_cast<unsigned long long*>(c);
  h->ws.cap_rows = rows;
  h->ws.cap_b = b;
  return SPECDEC_OK;
}

// Makes sure the workspace covers this call.  With a reservation that covers B,
// nothing is read back; the kernels check the row bound on the device.
int ensure_capacity(specdec_ctx* h, const int32_t* cu, int B, cudaStream_t stream) {
  if (h->reserved && B <= h->res_b) {
    if (h->ws.cap_rows < h->res_rows || h->ws.cap_b < h->res_b)
      return alloc_workspace(h, h->res_rows, h->res_b);
    return SPECDEC_OK;
  }
  int32_t nd = 0;
  if (cudaMemcpyAsync(&nd, cu + B, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return SPECDEC_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SPECDEC_ERR_CUDA;
  if (nd < 0) nd = 0;
  const int64_t rows = (int64_t)nd + B;
  if (rows > h->ws.cap_rows || B > h->ws.cap_b)
    return alloc_workspace(h, std::max(rows, h->ws.cap_rows), std::max(B, h->ws.cap_b));
  return SPECDEC_OK;
}

template <typename TT>
FusedConfig fused_config(specdec_ctx* h, int dtype, int V, const void* logits, const float* q) {
  FusedConfig f;
  const int esize = sizeof(TT);
  if (((int64_t)V * esize) % 16 != 0 || ((int64_t)V * 4) % 16 != 0) return f;
  if (reinterpret_cast<uintptr_t>(logits) % 16 != 0 || reinterpret_cast<uintptr_t>(q) % 16 != 0)
    return f;
  const int fixed = (int)round_up(sizeof(FusedShared), 128);
  for (int ci = 0; ci < 5; ++ci) {
    const int C = kClusterSizes[ci];
    const int L = (int)round_up((V + C - 1) / C, 8);
    const int tbytes = (int)round_up((int64_t)L * esize, 128);
    const int ring_room = h->smem_optin - tbytes - fixed;
    if (ring_room < kMinRing * kChunk * 4) continue;
    if ((L + kChunk - 1) / kChunk > kMaxChunks) continue;
    f.C = C;
    f.slice_len = L;
    f.tbuf_bytes = tbytes;
    f.nq = std::min(16, ring_room / (kChunk * 4));
    f.smem = tbytes + f.nq * kChunk * 4 + fixed;
    int& cs = h->occ_cache[dtype][ci][0];
    int& cn = h->occ_cache[dtype][ci][1];
    if (cs != f.smem) {
      auto kern = fused_row_kernel<TT>;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, f.smem) != cudaSuccess)
        return FusedConfig{};
      if (C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return FusedConfig{};
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(C * h->num_sms);
      cfg.blockDim = dim3(kFusedThreads);
      cfg.dynamicSmemBytes = f.smem;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = C;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return FusedConfig{};
      }
      cs = f.smem;
      cn = n;
    }
    f.clusters = cn;
    f.ok = true;
    return f;
  }
  return f;
}

template <typename TT>
int launch_sampling(specdec_ctx* h, Params& P, const FusedConfig& f, int path, cudaStream_t st) {
  const int B = P.B;
  if (h->ev_before) cudaEventRecord(h->ev_before, st);
  if (path == SPECDEC_PATH_PAIR) {
    const bool small = h->pair_threads == 256;
    auto kern = small ? pair_row_kernel<TT, 256> : pair_row_kernel<TT, 512>;
    int& nclus = h->pair_clusters[sizeof(TT) == 2][small];
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(h->pair_threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    if (nclus == 0) {
      cfg.gridDim = dim3(2 * h->num_sms);
      if (cudaOccupancyMaxActiveClusters(&nclus, kern, &cfg) != cudaSuccess || nclus <= 0) {
        cudaGetLastError();
        nclus = 0;
        return SPECDEC_ERR_CUDA;
      }
    }
    cfg.gridDim = dim3(2 * nclus);
    if (cudaLaunchKernelEx(&cfg, kern, P) != cudaSuccess) return SPECDEC_ERR_CUDA;
  } else if (path == SPECDEC_PATH_STREAM) {
    const int ctas = h->stream_ctas;
    const int fixed = (int)((sizeof(StreamShared) + 127) / 128 * 128);
    const int budget = ctas == 1 ? h->smem_optin : h->smem_per_sm / 2 - 1024;
    const int ns = std::min(kMaxStages, (budget - fixed) / kStageBytes);
    const int smem = ns * kStageBytes + fixed;
    P.nq = ns;
    auto kern = ctas == 1 ? stream_row_kernel<TT, 1> : stream_row_kernel<TT, 2>;
    int& cached = h->stream_smem[(sizeof(TT) == 2) * 2 + (ctas - 1)];
    if (cached != smem) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return SPECDEC_ERR_CUDA;
      cached = smem;
    }
    kern<<<h->num_sms * ctas, kStreamThreads, smem, st>>>(P);
  } else if (path == SPECDEC_PATH_DUAL) {
    dual_row_kernel<TT><<<h->num_sms * 2, 512, 0, st>>>(P);
  } else if (path == SPECDEC_PATH_SWEEP) {
    if (P.topk || P.topp) {
      const bool one = h->adj_threads == 1024;
      auto kern = one ? sweep_row_kernel<TT, 1024, 1, true> : sweep_row_kernel<TT, 512, 2, true>;
      int& set = h->adj_smem_set[sizeof(TT) == 2][one];
      if (!set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(AdjShared)) != cudaSuccess)
          return SPECDEC_ERR_CUDA;
        set = 1;
      }
      kern<<<h->num_sms * (one ? 1 : 2), one ? 1024 : 512, sizeof(AdjShared), st>>>(P);
    }
    else {
      // Draft rows given: two 512-thread CTAs per SM.  One-hot drafts: eight
      // 128-thread CTAs, so that while some CTAs draw a race (ALU work on a
      // row in L2) the others keep streaming rows from HBM.
      const int th = h->sweep_threads ? h->sweep_threads : (P.q ? 512 : 128);
      if (th == 512)
        sweep_row_kernel<TT, 512, 2><<<h->sweep_ctas ? h->sweep_ctas : h->num_sms * 2, 512, 0, st>>>(P);
      else if (th == 256)
        sweep_row_kernel<TT, 256, 4><<<h->num_sms * 4, 256, 0, st>>>(P);
      else if (th == 128)
        sweep_row_kernel<TT, 128, 8><<<h->num_sms * 8, 128, 0, st>>>(P);
      else if (th == 64)
        sweep_row_kernel<TT, 64, 16><<<h->num_sms * 16, 64, 0, st>>>(P);
      else
        sweep_row_kernel<TT, 1024, 1><<<h->num_sms, 1024, 0, st>>>(P);
    }
  } else if (path == SPECDEC_PATH_FUSED) {
    P.slice_len = f.slice_len;
    P.tbuf_bytes = f.tbuf_bytes;
    P.nq = f.nq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(f.C * f.clusters);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = f.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = f.C;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, fused_row_kernel<TT>, P) != cudaSuccess) return SPECDEC_ERR_CUDA;
  } else {
    const int grid = h->num_sms * 8;
    stats_kernel<TT><<<grid, kRowThreads, 0, st>>>(P);
    verify_kernel<TT><<<grid, kRowThreads, 0, st>>>(P);
  }
  if (h->ev_after) cudaEventRecord(h->ev_after, st);
  if (launch_dependent(finalize_kernel, (B + 255) / 256, 256, st, P) != cudaSuccess ||
      launch_dependent(race_kernel<TT>, h->num_sms * 8, kRowThreads, st, P) != cudaSuccess)
    return SPECDEC_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

template <typename TT>
int launch_greedy(specdec_ctx* h, Params& P, bool vec_ok, cudaStream_t st) {
  if (h->ev_before) cudaEventRecord(h->ev_before, st);
  greedy_partial_kernel<TT><<<h->num_sms * 8, kRowThreads, 0, st>>>(P, vec_ok ? 1 : 0);
  if (h->ev_after) cudaEventRecord(h->ev_after, st);
  if (launch_dependent(greedy_finalize_kernel, (P.B + 7) / 8, 256, st, P) != cudaSuccess)
    return SPECDEC_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

}  // namespace

extern "C" {

int specdec_create(specdec_handle_t* out, int device) {
  if (!out) return SPECDEC_ERR_INVALID_ARG;
  *out = nullptr;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess) {
    cudaGetLastError();
    return SPECDEC_ERR_CUDA;
  }
  if (device < 0 || device >= n) return SPECDEC_ERR_INVALID_ARG;
  DeviceGuard guard(device);
  if (!guard.ok()) return SPECDEC_ERR_CUDA;
  specdec_ctx* h = new (std::nothrow) specdec_ctx();
  if (!h) return SPECDEC_ERR_OOM;
  h->device = device;
  cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device);
  cudaDeviceGetAttribute(&h->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  cudaDeviceGetAttribute(&h->smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device);
  // tuning knobs for measurements: sweep block size (1024 .. 64) and grid, adjusted sweep block
  // size (512, 1024), pair block size (512, 256) and stream CTAs per SM
  if (const char* e = std::getenv("SPECDEC_SWEEP_THREADS")) {
    const int v = std::atoi(e);
    if (v == 64 || v == 128 || v == 256 || v == 512 || v == 1024) h->sweep_threads = v;
  }
  if (const char* e = std::getenv("SPECDEC_SWEEP_CTAS")) {
    const int v = std::atoi(e);
    if (v >= 1 && v <= 2 * h->num_sms) h->sweep_ctas = v;
  }
  if (const char* e = std::getenv("SPECDEC_ADJ_THREADS")) {
    const int v = std::atoi(e);
    if (v == 512 || v == 1024) h->adj_threads = v;
  }
  if (const char* e = std::getenv("SPECDEC_PAIR_THREADS")) {
    const int v = std::atoi(e);
    if (v == 256 || v == 512) h->pair_threads = v;
  }
  if (const char* e = std::getenv("SPECDEC_STREAM_CTAS")) {
    const int v = std::atoi(e);
    if (v == 1 || v == 2) h->stream_ctas = v;
  }
  if (cudaMalloc(&h->small, 64) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return SPECDEC_ERR_OOM;
  }
  if (cudaMemset(h->small, 0, 64) != cudaSuccess) {
    cudaFree(h->small);
    delete h;
    return SPECDEC_ERR_CUDA;
  }
  *out = h;
  return SPECDEC_OK;
}

int specdec_reserve(specdec_handle_t h, int64_t max_draft_positions, int max_batch) {
  if (!h || max_draft_positions < 0 || max_batch <= 0) return SPECDEC_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok()) return SPECDEC_ERR_CUDA;
  h->reserved = true;
  h->res_rows = max_draft_positions + max_batch;
  h->res_b = max_batch;
  if (h->ws.cap_rows >= h->res_rows && h->ws.cap_b >= h->res_b) return SPECDEC_OK;
  return alloc_workspace(h, h->res_rows, h->res_b);
}

int specdec_rejection_sample_topk_topp(
    specdec_handle_t h, const void* target_logits, int dtype, const float* draft_probs,
    const int32_t* draft_ids, const int32_t* cu_num_draft_tokens, int B, int V, float T,
    const int32_t* top_k, const float* top_p, uint64_t seed, uint64_t request_offset,
    int32_t* out_tokens, int32_t* out_num_accepted, float* out_beta, float* out_target_prob,
    float* out_draft_prob, int32_t* out_accept, void* stream) {
  if (!h) return SPECDEC_ERR_INVALID_ARG;
  if (dtype != SPECDEC_F32 && dtype != SPECDEC_BF16) return SPECDEC_ERR_UNSUPPORTED_DTYPE;
  if (B <= 0 || V <= 0 || V > (1 << 30)) return SPECDEC_ERR_INVALID_ARG;
  if (!std::isfinite(T) || T < 0.0f) return SPECDEC_ERR_INVALID_ARG;
  if (!target_logits || !draft_ids || !cu_num_draft_tokens || !out_tokens || !out_num_accepted)
    return SPECDEC_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok()) return SPECDEC_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = ensure_capacity(h, cu_num_draft_tokens, B, st);
  if (rc != SPECDEC_OK) return rc;

  Params P = {};
  P.logits = target_logits;
  P.q = draft_probs;
  P.ids = draft_ids;
  P.cu = cu_num_draft_tokens;
  P.B = B;
  P.V = V;
  P.c = T > 0.0f ? kLog2e / T : 0.0f;
  P.seed = seed;
  P.req_offset = request_offset;
  P.epoch = ++h->epoch;
  P.out_tokens = out_tokens;
  P.out_nacc = out_num_accepted;
  P.out_beta = out_beta;
  P.out_px = out_target_prob;
  P.out_qx = out_draft_prob;
  P.out_acc = out_accept;
  P.row_stats = h->ws.row_stats;
  P.status = h->ws.status;
  P.gkeys = h->ws.gkeys;
  P.ws_nacc = h->ws.ws_nacc;
  P.defer_list = h->ws.defer_list;
  P.rpart = h->ws.rpart;
  P.rcount = h->ws.rcount;
  P.dual_part = h->ws.dual_part;
  P.dual_cnt = h->ws.dual_cnt;
  P.dual_skip = h->ws.dual_skip;
  P.dual_race = h->ws.dual_race;
  P.topk = T > 0.0f ? top_k : nullptr;   // the greedy path keeps the argmax either way
  P.topp = T > 0.0f ? top_p : nullptr;
  P.row_tau = (P.topk || P.topp) ? h->ws.row_tau : nullptr;
  P.adj_ctr = h->adj_ctr;
  P.rslices = (int)std::min<int64_t>(
      kRaceMaxSlices, std::max<int64_t>(1, (V + kRaceSliceTarget - 1) / kRaceSliceTarget));
  P.rslice_len = (int)round_up((V + P.rslices - 1) / P.rslices, 8);
  P.rstride = kRaceMaxSlices;
  P.defer_count = reinterpret_cast<int32_t*>(h->small + 1);
  P.err = h->small;
  P.cap_rows = h->ws.cap_rows;
  P.cap_b = h->ws.cap_b;
  if (B > h->ws.cap_b) return SPECDEC_ERR_CAPACITY;

  const int esize = dtype == SPECDEC_BF16 ? 2 : 4;
  if (T == 0.0f) {
    const bool vec_ok = ((int64_t)V * esize) % 16 == 0 &&
                        reinterpret_cast<uintptr_t>(target_logits) % 16 == 0;
    h->last_path = SPECDEC_PATH_GREEDY;
    h->last_cluster = 0;
    return dtype == SPECDEC_BF16 ? launch_greedy<__nv_bfloat16>(h, P, vec_ok, st)
                                 : launch_greedy<float>(h, P, vec_ok, st);
  }
  P.vec_ok = ((int64_t)V * esize) % 16 == 0 && ((int64_t)V * 4) % 16 == 0 &&
             reinterpret_cast<uintptr_t>(target_logits) % 16 == 0 &&
             reinterpret_cast<uintptr_t>(draft_probs) % 16 == 0;
  P.sched = reinterpret_cast<unsigned long long*>(h->small + 2);
  P.wait_ns = h->fault_wait_ns;
  P.stall_peer = h->fault_mode == SPECDEC_FAULT_PAIR_STALL ? 1 : 0;
  // AUTO: with fewer requests than sweep CTAs (2 per SM), the sweep kernel's
  // later rows of a request usually decide before its earlier rows finish and
  // their races go to the race kernel; the pair kernel holds half as many rows
  // in flight, so it keeps them ahead (and halves the rows live in L2)
  int path = h->path_override;
  if (path == SPECDEC_PATH_AUTO) path = B < 2 * h->num_sms ? SPECDEC_PATH_PAIR : SPECDEC_PATH_SWEEP;
  if (!draft_probs) path = SPECDEC_PATH_SWEEP;  // one-hot drafts: the sweep kernel handles them
  if (P.topk || P.topp) path = SPECDEC_PATH_SWEEP;  // so do adjusted (top-k / top-p) rows
  if (path == SPECDEC_PATH_STREAM && !P.vec_ok) path = SPECDEC_PATH_SWEEP;
  FusedConfig f;
  if (path == SPECDEC_PATH_FUSED) {
    f = dtype == SPECDEC_BF16 ? fused_config<__nv_bfloat16>(h, dtype, V, target_logits, draft_probs)
                              : fused_config<float>(h, dtype, V, target_logits, draft_probs);
    if (!f.ok) path = SPECDEC_PATH_SWEEP;
  }
  h->last_path = path;
  h->last_cluster = path == SPECDEC_PATH_FUSED ? f.C : (path == SPECDEC_PATH_PAIR ? 2 : 0);
  return dtype == SPECDEC_BF16 ? launch_sampling<__nv_bfloat16>(h, P, f, path, st)
                               : launch_sampling<float>(h, P, f, path, st);
}

int specdec_rejection_sample_ex(specdec_handle_t h, const void* target_logits, int dtype,
                                const float* draft_probs, const int32_t* draft_ids,
                                const int32_t* cu_num_draft_tokens, int B, int V, float T,
                                uint64_t seed, uint64_t request_offset, int32_t* out_tokens,
                                int32_t* out_num_accepted, float* out_beta,
                                float* out_target_prob, float* out_draft_prob,
                                int32_t* out_accept, void* stream) {
  return specdec_rejection_sample_topk_topp(h, target_logits, dtype, draft_probs, draft_ids,
                                            cu_num_draft_tokens, B, V, T, nullptr, nullptr, seed,
                                            request_offset, out_tokens, out_num_accepted, out_beta,
                                            out_target_prob, out_draft_prob, out_accept, stream);
}

int specdec_rejection_sample(specdec_handle_t h, const void* target_logits, int dtype,
                             const float* draft_probs, const int32_t* draft_ids,
                             const int32_t* cu_num_draft_tokens, int B, int V, float T,
                             uint64_t seed, int32_t* out_tokens, int32_t* out_num_accepted,
                             float* out_beta, void* stream) {
  return specdec_rejection_sample_ex(h, target_logits, dtype, draft_probs, draft_ids,
                                     cu_num_draft_tokens, B, V, T, seed, 0, out_tokens,
                                     out_num_accepted, out_beta, nullptr, nullptr, nullptr, stream);
}

int specdec_tree_verify(specdec_handle_t h, const void* target_logits, int dtype,
                        const float* draft_probs, const int32_t* node_tokens,
                        const int32_t* node_parent, const int32_t* cu_num_nodes, int B, int V,
                        float T, uint64_t seed, uint64_t request_offset, int32_t* out_tokens,
                        int32_t* out_num_accepted, int32_t* out_path, void* stream) {
  if (!h) return SPECDEC_ERR_INVALID_ARG;
  if (dtype != SPECDEC_F32 && dtype != SPECDEC_BF16) return SPECDEC_ERR_UNSUPPORTED_DTYPE;
  if (B <= 0 || V <= 0 || V > (1 << 30)) return SPECDEC_ERR_INVALID_ARG;
  if (!std::isfinite(T) || T < 0.0f) return SPECDEC_ERR_INVALID_ARG;
  if (!target_logits || !node_tokens || !node_parent || !cu_num_nodes || !out_tokens ||
      !out_num_accepted || (T > 0.0f && !draft_probs))
    return SPECDEC_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok()) return SPECDEC_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TreeArgs a = {};
  a.logits = target_logits;
  a.q = T > 0.0f ? draft_probs : nullptr;
  a.tok = node_tokens;
  a.par = node_parent;
  a.cu = cu_num_nodes;
  a.B = B;
  a.V = V;
  a.c = T > 0.0f ? kLog2e / T : 0.0f;
  a.seed = seed;
  a.req_offset = request_offset;
  a.out_tokens = out_tokens;
  a.out_nacc = out_num_accepted;
  a.out_path = out_path;
  a.err = h->small;
  a.counter = reinterpret_cast<unsigned long long*>(h->small + 4);
  const int esize = dtype == SPECDEC_BF16 ? 2 : 4;
  a.vec_ok = ((int64_t)V * esize) % 16 == 0 && ((int64_t)V * 4) % 16 == 0 &&
             reinterpret_cast<uintptr_t>(target_logits) % 16 == 0 &&
             reinterpret_cast<uintptr_t>(a.q) % 16 == 0;
  if (h->ev_before) cudaEventRecord(h->ev_before, st);
  const int rc = launch_tree(a, dtype, h->num_sms, st);
  if (h->ev_after) cudaEventRecord(h->ev_after, st);
  return rc;
}

int specdec_get_error(specdec_handle_t h, int* device_error, void* stream) {
  if (!h || !device_error) return SPECDEC_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok()) return SPECDEC_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, h->small, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(h->small, 0, sizeof(uint32_t), st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return SPECDEC_ERR_CUDA;
  *device_error = (int)v;
  return SPECDEC_OK;
}

int specdec_set_path(specdec_handle_t h, int path) {
  if (!h || path < SPECDEC_PATH_AUTO || path > SPECDEC_PATH_DUAL || path == SPECDEC_PATH_GREEDY)
    return SPECDEC_ERR_INVALID_ARG;
  h->path_override = path;
  return SPECDEC_OK;
}

int specdec_set_timing_events(specdec_handle_t h, void* before_rows, void* after_rows) {
  if (!h || (before_rows == nullptr) != (after_rows == nullptr)) return SPECDEC_ERR_INVALID_ARG;
  h->ev_before = static_cast<cudaEvent_t>(before_rows);
  h->ev_after = static_cast<cudaEvent_t>(after_rows);
  return SPECDEC_OK;
}

int specdec_set_adjust_counters(specdec_handle_t h, uint64_t* device_counters) {
  if (!h) return SPECDEC_ERR_INVALID_ARG;
  h->adj_ctr = reinterpret_cast<unsigned long long*>(device_counters);
  return SPECDEC_OK;
}

int specdec_set_fault_injection(specdec_handle_t h, int mode, uint64_t wait_limit_ns) {
  if (!h || (mode != SPECDEC_FAULT_NONE && mode != SPECDEC_FAULT_PAIR_STALL))
    return SPECDEC_ERR_INVALID_ARG;
  if (mode != SPECDEC_FAULT_NONE && (wait_limit_ns == 0 || wait_limit_ns > 2000000000ull))
    return SPECDEC_ERR_INVALID_ARG;
  h->fault_mode = mode;
  h->fault_wait_ns = mode == SPECDEC_FAULT_NONE ? 0 : wait_limit_ns;
  return SPECDEC_OK;
}

int specdec_last_path(specdec_handle_t h, int* path, int* cluster_size) {
  if (!h) return SPECDEC_ERR_INVALID_ARG;
  if (path) *path = h->last_path;
  if (cluster_size) *cluster_size = h->last_cluster;
  return SPECDEC_OK;
}

int specdec_uniform(uint64_t seed, uint64_t b, uint64_t pos, uint32_t stream_id, uint64_t v0,
                    int64_t n, float* out, void* stream) {
  if (n < 0 || (n > 0 && !out)) return SPECDEC_ERR_INVALID_ARG;
  if (n == 0) return SPECDEC_OK;
  const uint64_t key = stream_key(seed, b, pos, stream_id);
  const int grid = (int)std::min<int64_t>((n + 255) / 256, 4096);
  uniform_fill_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(key, v0, n, out);
  return cudaGetLastError() == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

int specdec_neg_log_uniform(uint32_t k0, int64_t n, float* out, void* stream) {
  if (n < 0 || (n > 0 && !out) || (int64_t)k0 + n > (int64_t)(1u << 23)) return SPECDEC_ERR_INVALID_ARG;
  if (n == 0) return SPECDEC_OK;
  const int grid = (int)std::min<int64_t>((n + 255) / 256, 4096);
  neglog_fill_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(k0, n, out);
  return cudaGetLastError() == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

int specdec_selection_mass(const float* z, int64_t n, int V, uint64_t* out_mass, float* out_pow2,
                           void* stream) {
  if (n < 0 || V <= 0 || V > (1 << 30) || (n > 0 && (!z || (!out_mass && !out_pow2))))
    return SPECDEC_ERR_INVALID_ARG;
  if (n == 0) return SPECDEC_OK;
  const int grid = (int)std::min<int64_t>((n + 255) / 256, 4096);
  selection_mass_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      z, n, V, reinterpret_cast<unsigned long long*>(out_mass), out_pow2);
  return cudaGetLastError() == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

const char* specdec_status_string(int status) {
  switch (status) {
    case SPECDEC_OK: return "ok";
    case SPECDEC_ERR_INVALID_ARG: return "invalid argument";
    case SPECDEC_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case SPECDEC_ERR_CUDA: return "CUDA error";
    case SPECDEC_ERR_OOM: return "out of device memory";
    case SPECDEC_ERR_BAD_DRAFT_ID: return "draft id outside [0, V)";
    case SPECDEC_ERR_CAPACITY: return "batch larger than the workspace";
    case SPECDEC_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int specdec_destroy(specdec_handle_t h) {
  if (!h) return SPECDEC_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  cudaDeviceSynchronize();
  free_workspace(h);
  if (h->small) cudaFree(h->small);
  delete h;
  return SPECDEC_OK;
}

}  // extern "C"
