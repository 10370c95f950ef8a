// Verifier kernels.
//
//   sweep_row_kernel   the default row kernel (T > 0): persistent, 2 CTAs of 512
//                      threads per SM, one target row per CTA at a time.  Sweep 1
//                      streams the target row from HBM for (max, sum); sweep 2
//                      re-reads it from L2 with the draft row for beta, the accept
//                      test and, when the request's earlier rows are known to be
//                      accepted, the exponential race of the extra token.  With
//                      kAdj, requests may carry top-k / top-p: a threshold
//                      selection runs between the sweeps (the adjusted-row section).
//   pair_row_kernel    the same sweeps with each row split over a 2-CTA cluster
//                      ((max, sum) and partials exchanged in distributed shared
//                      memory); the default for small batches.
//   dual_row_kernel    two independent CTAs per row (each sweeps the whole row for
//                      (max, sum) and half of it for the rest), no waiting.
//   stream_row_kernel  the sweeps fed by bulk copies through a shared-memory ring.
//   fused_row_kernel   one HBM pass per (target row, draft row) pair: a cluster of
//                      C CTAs holds the target row in shared memory.
//   stats_kernel +     the two-pass form, for any layout.
//   verify_kernel
//   finalize_kernel    per-request first-rejection scan over cu_num_draft_tokens.
//   race_kernel        the race for requests whose extra token the row kernel could
//                      not draw (its row ran before the earlier rows of the request
//                      finished): re-reads that single row, in slices.
//   greedy_*           T = 0: argmax per row (warp items, 64-bit atomicMax), then
//                      the scan.
//
// Method: Algorithm 1 and Section 2.3 of Leviathan et al. as restated on the
// bloss0m and vllbc reading-notes pages; accept test r < min(1, p/q) as in the
// timinsight guide's Step 2 pseudo-code; beta from Theorem 3.5.
#pragma once

// Non-template kernels are `static`: each translation unit that launches them
// (the handle path and the allocation-free path) keeps its own copy.

#include "device_common.cuh"

namespace specdec {

// ---------------------------------------------------------------------------
// Shared parameter block.
// ---------------------------------------------------------------------------
struct Params {
  const void* logits;      // [N_t, V] float or bf16
  const float* q;          // [N_d, V] or null (greedy)
  const int32_t* ids;      // [N_d]
  const int32_t* cu;       // [B+1]
  int B;
  int V;
  float c;                 // log2(e) / T
  uint64_t seed;
  uint64_t req_offset;     // generator request index = req_offset + b
  uint64_t epoch;          // call counter (status words of this call carry it)
  int32_t* out_tokens;     // [N_t]
  int32_t* out_nacc;       // [B]
  float* out_beta;         // [N_d] or null
  float* out_px;           // [N_d] or null
  float* out_qx;           // [N_d] or null
  int32_t* out_acc;        // [N_d] or null
  // workspace
  float2* row_stats;       // [cap_rows] (max, sum) of each target row
  uint64_t* status;        // [cap_rows]
  uint64_t* gkeys;         // [cap_rows] greedy argmax key per row (0 between calls)
  int32_t* ws_nacc;        // [cap_B] n_b for the race kernel
  int32_t* defer_list;     // [cap_B]
  int32_t* defer_count;    // [1]
  float4* rpart;           // [cap_B * rstride] partial race winners per deferred request
  int32_t* rcount;         // [cap_B] slices finished per deferred request (reset by the last one)
  int rslices;             // slices per deferred row
  int rslice_len;          // elements per slice (multiple of 8)
  int rstride;             // rpart entries per deferred request (>= rslices)
  unsigned long long* sched;  // [1] next work slot of the sweep kernel (reset by finalize)
  const int32_t* topk;     // [B] per-request top-k or null (adjusted rows, sweep kernel only)
  const float* topp;       // [B] per-request top-p or null
  float* row_tau;          // [cap_rows] logit threshold of each adjusted row, or null
  unsigned long long* adj_ctr;  // [kAdjCounters] selection statistics (profiling), or null
  float4* dual_part;       // [2 cap_rows] dual kernel: each half's (beta, race w, e, index)
  int32_t* dual_cnt;       // [cap_rows] dual kernel: halves done (0 between calls)
  unsigned long long* dual_skip;  // [cap_rows] dual kernel: bonus-row skip decision (epoch-tagged)
  unsigned long long* dual_race;  // [cap_rows] dual kernel: race decision (epoch-tagged)
  uint32_t* err;           // [1] sticky device error word
  int64_t cap_rows;
  int cap_b;
  // fused kernel geometry
  int slice_len;           // elements per cluster rank (multiple of 8)
  int tbuf_bytes;          // bytes of the target slice buffer (rank 0, 128-aligned)
  int nq;                  // draft ring stages
  int vec_ok;              // rows are 16-byte aligned: vector loads allowed
  // test hook (specdec_set_fault_injection): the pair kernel's bounded waits
  // give up after wait_ns (0: the default 2 s), and with stall_peer its rank 0
  // withholds the first work slot from rank 1, whose wait then runs out
  uint64_t wait_ns;
  int stall_peer;
};

constexpr int kChunk = 4096;          // elements per bulk copy / pipeline step
constexpr int kRaceMaxSlices = 64;    // a deferred row is split over at most this many CTAs
constexpr int kRaceSliceTarget = 4096; // elements per slice the split aims at
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kFusedThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxCluster = 16;
constexpr int kMaxChunks = 64;

__device__ __forceinline__ void set_err(uint32_t* err, uint32_t bits) { atomicOr(err, bits); }

// Kernels launched as programmatic dependents (launch_dependent below) start
// while the previous kernel in the stream drains and wait here, before their
// first read of its results, until it has completed and its writes are visible.
__device__ __forceinline__ void wait_for_previous_kernel() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launches kern<<<grid, block, 0, st>>>(args...) as a programmatic dependent of
// the previous kernel on st: its launch and block placement overlap that
// kernel's tail; the kernel itself must call wait_for_previous_kernel() first.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), int grid, int block, cudaStream_t st,
                                    Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---------------------------------------------------------------------------
// Fused single-pass row kernel (T > 0).
// ---------------------------------------------------------------------------
struct alignas(16) FusedShared {
  uint64_t tfull[kMaxChunks];
  uint64_t tempty[kMaxChunks];
  uint64_t qfull[16];
  uint64_t qempty[16];
  uint64_t x1full[2];
  uint64_t x2full[2];
  float4 xch1[2][kMaxCluster];   // (max, sum, prefix state, -) from every rank
  float4 xch2[2][kMaxCluster];   // (beta, race w, race e, race index) at rank 0
  float4 red[2][kConsumerWarps];
  int gmax;
  int bad;
  volatile int abort_flag;
};

template <typename TT>
__global__ void __launch_bounds__(kFusedThreads, 1) fused_row_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  constexpr int kEl = 16 / sizeof(TT);  // elements per 16-byte target vector
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t C = cluster_nctarank();
  const uint32_t cid = cluster_id_x();
  const uint32_t ncl = ncluster_x();

  TT* tbuf = reinterpret_cast<TT*>(smem_raw);
  float* qring = reinterpret_cast<float*>(smem_raw + P.tbuf_bytes);
  FusedShared& S = *reinterpret_cast<FusedShared*>(smem_raw + P.tbuf_bytes +
                                                   (size_t)P.nq * kChunk * sizeof(float));

  const int V = P.V, B = P.B;
  const int s0 = min((int)rank * P.slice_len, V);
  const int s1 = min(s0 + P.slice_len, V);
  const int slen = s1 - s0;
  const int nch = (slen + kChunk - 1) / kChunk;

  // ---- prologue: barriers, scan of cu (largest gamma, validity) ----------
  if (tid == 0) {
    for (int j = 0; j < nch; ++j) {
      mbar_init(smem_addr(&S.tfull[j]), 1);
      mbar_init(smem_addr(&S.tempty[j]), kConsumerWarps);
    }
    for (int s = 0; s < P.nq; ++s) {
      mbar_init(smem_addr(&S.qfull[s]), 1);
      mbar_init(smem_addr(&S.qempty[s]), kConsumerWarps);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(smem_addr(&S.x1full[p]), C);
      mbar_init(smem_addr(&S.x2full[p]), C);
    }
    S.gmax = 0;
    S.bad = 0;
    S.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  {
    int gm = 0, bad = 0;
    for (int b = tid; b < B; b += blockDim.x) {
      int g = __ldg(P.cu + b + 1) - __ldg(P.cu + b);
      gm = max(gm, g);
      bad |= (g < 0);
    }
    if (gm) atomicMax(&S.gmax, gm);
    if (bad) atomicOr(&S.bad, 1);
  }
  cluster_sync_all();  // barrier inits visible cluster-wide; gmax / bad final
  if (cid == 0 && rank == 0 && tid == 0) {
    if (S.bad || __ldg(P.cu) != 0) set_err(P.err, SPECDEC_DEVERR_BAD_CU);
    if (P.defer_count) *P.defer_count = 0;
  }
  const int gmax = S.gmax;
  const int64_t total_slots = (int64_t)B * (gmax + 1);

  if (warp == kConsumerWarps) {
    // ===================== producer warp ====================================
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      uint32_t uc = 0, qc = 0;
      uint32_t t_issued[kMaxChunks];
      uint32_t q_issued[16];
      for (int j = 0; j < nch; ++j) t_issued[j] = 0;
      for (int s = 0; s < P.nq; ++s) q_issued[s] = 0;
      for (int64_t u = cid; u < total_slots && !S.abort_flag; u += ncl) {
        const int i = (int)(u / B), b = (int)(u % B);
        const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
        if (i > g) continue;
        const int64_t t = (int64_t)c0 + b + i;
        if (t >= P.cap_rows) continue;
        const bool has_q = i < g;
        const TT* trow = reinterpret_cast<const TT*>(P.logits) + t * (int64_t)V + s0;
        for (int j = 0; j < nch; ++j) {
          if (!mbar_wait(smem_addr(&S.tempty[j]), (uc & 1) ^ 1)) {
            S.abort_flag = 1;
            break;
          }
          const int n = min(kChunk, slen - j * kChunk);
          mbar_arrive_expect_tx(smem_addr(&S.tfull[j]), n * sizeof(TT));
          bulk_load(smem_addr(tbuf + j * kChunk), trow + j * kChunk, n * sizeof(TT),
                    smem_addr(&S.tfull[j]), pol);
          ++t_issued[j];
        }
        if (has_q && !S.abort_flag) {
          const float* qrow = P.q + ((int64_t)c0 + i) * (int64_t)V + s0;
          for (int j = 0; j < nch; ++j, ++qc) {
            const int s = qc % P.nq;
            if (!mbar_wait(smem_addr(&S.qempty[s]), ((qc / P.nq) & 1) ^ 1)) {
              S.abort_flag = 1;
              break;
            }
            const int n = min(kChunk, slen - j * kChunk);
            mbar_arrive_expect_tx(smem_addr(&S.qfull[s]), n * 4);
            bulk_load(smem_addr(qring + (size_t)s * kChunk), qrow + j * kChunk, n * 4,
                      smem_addr(&S.qfull[s]), pol);
            ++q_issued[s];
          }
        }
        ++uc;
      }
      if (S.abort_flag) {
        // Let every copy this CTA issued land before the CTA can exit.
        set_err(P.err, SPECDEC_DEVERR_TIMEOUT);
        for (int j = 0; j < nch; ++j)
          if (t_issued[j]) mbar_wait(smem_addr(&S.tfull[j]), (t_issued[j] - 1) & 1);
        for (int s = 0; s < P.nq; ++s)
          if (q_issued[s]) mbar_wait(smem_addr(&S.qfull[s]), (q_issued[s] - 1) & 1);
      }
    }
    __syncwarp();
  } else {
    // ===================== consumer warps ===================================
    uint32_t uc = 0, qc = 0;
    for (int64_t u = cid; u < total_slots; u += ncl) {
      const int i = (int)(u / B), b = (int)(u % B);
      const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
      if (i > g) continue;
      const int64_t t = (int64_t)c0 + b + i;
      if (t >= P.cap_rows) {
        if (tid == 0 && rank == 0) set_err(P.err, SPECDEC_DEVERR_CAPACITY);
        continue;
      }
      const int64_t d = (int64_t)c0 + i;
      const bool has_q = i < g;
      const int par = uc & 1;
      bool ok = true;

      // ---- pass 1: (max, sum) of this rank's slice ---------------------------
      float m = -INFINITY, s = 0.0f;
      for (int j = 0; j < nch; ++j) {
        ok &= S.abort_flag ? false : mbar_wait(smem_addr(&S.tfull[j]), uc & 1);
        const int n = min(kChunk, slen - j * kChunk);
        const TT* ch = tbuf + j * kChunk;
        for (int e = tid * kEl; e < n; e += kConsumers * kEl) {
          float x[kEl];
          if constexpr (sizeof(TT) == 2) {
            uint4 w = *reinterpret_cast<const uint4*>(ch + e);
            x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
            x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
          } else {
            float4 w = *reinterpret_cast<const float4*>(ch + e);
            x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
          }
          float vm = x[0];
#pragma unroll
          for (int k = 1; k < kEl; ++k) vm = fmaxf(vm, x[k]);
          if (vm > m) {
            s *= ex2((m - vm) * P.c);
            m = vm;
          }
          if (m != -INFINITY) {
            float acc = 0.0f;
#pragma unroll
            for (int k = 0; k < kEl; ++k) acc += ex2((x[k] - m) * P.c);
            s += acc;
          }
        }
      }
      warp_softmax(m, s, P.c);
      if (lane == 0) S.red[par][warp] = make_float4(m, s, 0.f, 0.f);
      named_bar_sync(1, kConsumers);
      m = -INFINITY;
      s = 0.0f;
      for (int w = 0; w < kConsumerWarps; ++w) softmax_merge(m, s, S.red[par][w].x, S.red[par][w].y, P.c);

      // ---- exchange 1: every rank gets every rank's (max, sum) --------------
      if (tid == 0) {
        int prefix = kPrefixAllAccepted;
        if (rank == 0 && i > 0) prefix = read_prefix(P.status, t - i, i, P.epoch);
        const uint32_t slot = smem_addr(&S.xch1[par][rank]);
        for (uint32_t r = 0; r < C; ++r) {
          st_cluster_v4(mapa(slot, r), m, s, __int_as_float(prefix), 0.f);
          mbar_arrive_cluster(mapa(smem_addr(&S.x1full[par]), r));
        }
      }
      ok &= S.abort_flag ? false : mbar_wait_cluster(smem_addr(&S.x1full[par]), (uc >> 1) & 1);
      float M = -INFINITY, Ssum = 0.0f;
      for (uint32_t r = 0; r < C; ++r) softmax_merge(M, Ssum, S.xch1[par][r].x, S.xch1[par][r].y, P.c);
      const int prefix = __float_as_int(S.xch1[par][0].z);
      const float invS = 1.0f / Ssum;

      // ---- accept test (identical in every thread of every rank) -------------
      int x = -1;
      float px = 0.0f, qx = 0.0f;
      bool acc = false, valid = true;
      if (has_q) {
        x = __ldg(P.ids + d);
        valid = (x >= 0 && x < V);
        if (valid) {
          const float lx = load_logit(reinterpret_cast<const TT*>(P.logits) + t * (int64_t)V + x);
          px = ex2((lx - M) * P.c) * invS;
          qx = __ldg(P.q + d * (int64_t)V + x);
        }
        const float r = uniform_from_bits(uniform_bits(stream_key(P.seed, P.req_offset + b, i, 0), 0));
        acc = accept_test(r, px, qx);
      }
      const bool race = (prefix == kPrefixAllAccepted) && (!has_q || !acc);
      const bool resid = has_q && !acc;
      const uint64_t rkey = stream_key(P.seed, P.req_offset + b, i, 1);

      // ---- pass 2: beta and the race over the slice -------------------------
      float beta = 0.0f;
      Race best = race_none();
      for (int j = 0; j < nch; ++j) {
        const int n = min(kChunk, slen - j * kChunk);
        int st = 0;
        if (has_q) {
          st = qc % P.nq;
          ok &= S.abort_flag ? false : mbar_wait(smem_addr(&S.qfull[st]), (qc / P.nq) & 1);
        }
        if (has_q || race) {
          const TT* ch = tbuf + j * kChunk;
          const float* qch = qring + (size_t)st * kChunk;
          for (int e = tid * 4; e < n; e += kConsumers * 4) {
            float l[4];
            if constexpr (sizeof(TT) == 2) {
              uint2 w = *reinterpret_cast<const uint2*>(ch + e);
              l[0] = bf16_lo(w.x); l[1] = bf16_hi(w.x); l[2] = bf16_lo(w.y); l[3] = bf16_hi(w.y);
            } else {
              float4 w = *reinterpret_cast<const float4*>(ch + e);
              l[0] = w.x; l[1] = w.y; l[2] = w.z; l[3] = w.w;
            }
            float p[4], qv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 4; ++k) p[k] = ex2((l[k] - M) * P.c) * invS;
            if (has_q) {
              float4 w = *reinterpret_cast<const float4*>(qch + e);
              qv[0] = w.x; qv[1] = w.y; qv[2] = w.z; qv[3] = w.w;
              beta += (fminf(p[0], qv[0]) + fminf(p[1], qv[1])) +
                      (fminf(p[2], qv[2]) + fminf(p[3], qv[3]));
            }
            if (race) {
              const int v0 = s0 + j * kChunk + e;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                race_offer(best, resid ? fmaxf(p[k] - qv[k], 0.0f) : p[k], rkey, (uint32_t)(v0 + k));
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_addr(&S.tempty[j]));
          if (has_q) mbar_arrive(smem_addr(&S.qempty[st]));
        }
        if (has_q) ++qc;
      }
      beta = warp_sum(beta);
      warp_race(best);
      if (lane == 0) S.red[par ^ 1][warp] = make_float4(beta, best.w, best.e, __int_as_float(best.idx));
      named_bar_sync(1, kConsumers);

      // ---- exchange 2: partial beta / race to rank 0, which writes outputs ---
      if (tid == 0) {
        float bsum = 0.0f;
        Race cb = race_none();
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float4 r4 = S.red[par ^ 1][w];
          bsum += r4.x;
          race_merge(cb, r4.y, r4.z, __float_as_int(r4.w));
        }
        st_cluster_v4(mapa(smem_addr(&S.xch2[par][rank]), 0), bsum, cb.w, cb.e, __int_as_float(cb.idx));
        mbar_arrive_cluster(mapa(smem_addr(&S.x2full[par]), 0));
        if (rank == 0) {
          ok &= S.abort_flag ? false : mbar_wait_cluster(smem_addr(&S.x2full[par]), (uc >> 1) & 1);
          float btot = 0.0f;
          Race tb = race_none();
          for (uint32_t r = 0; r < C; ++r) {
            const float4 r4 = S.xch2[par][r];
            btot += r4.x;
            race_merge(tb, r4.y, r4.z, __float_as_int(r4.w));
          }
          if (ok) {
            P.row_stats[t] = make_float2(M, Ssum);
            uint32_t flags = kStDone;
            if (has_q) {
              if (!valid) set_err(P.err, SPECDEC_DEVERR_BAD_DRAFT_ID);
              if (acc) flags |= kStAccepted;
              if (P.out_beta) P.out_beta[d] = btot;
              if (P.out_px) P.out_px[d] = px;
              if (P.out_qx) P.out_qx[d] = qx;
              if (P.out_acc) P.out_acc[d] = acc ? 1 : 0;
            }
            if (race && tb.w > 0.0f) {
              P.out_tokens[t] = tb.idx;
              flags |= kStRaceDone;
            }
            st_relaxed_u64(P.status + t, make_status(P.epoch, flags));
          }
        }
      }
      ++uc;
      if (named_bar_or(1, kConsumers, !ok || S.abort_flag)) {
        S.abort_flag = 1;
        if (tid == 0) set_err(P.err, SPECDEC_DEVERR_TIMEOUT);
        break;
      }
    }
  }
  __syncwarp();
  cluster_sync_all();  // no rank leaves while a peer may still touch its shared memory
}

// ---------------------------------------------------------------------------
// Sweep row kernel (T > 0): one CTA per SM, one (target row, draft row) pair at
// a time.  Sweep 1 reads the target row from HBM (L2 evict_last) for (max, sum);
// sweep 2 reads it again, now from L2 (evict_first), together with the draft
// row (evict_first) for beta, the accept test and the race.  About one target
// row per SM is live in L2 at a time (~78 MB for V = 256000 bf16).  Work slots
// are taken in position-major order (every request's position 0, then every
// position 1, ...) from a global counter, so the earlier rows of a request are
// usually finished when a later row starts: the row that turns out to be the
// request's first rejection (or the bonus row after all drafts were accepted)
// draws the extra token in the same sweep, and a bonus row whose request already
// rejected a draft is not read at all.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg_hint(const void* p, uint64_t pol) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "l"(pol));
  return r;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

template <typename TT>
__device__ __forceinline__ void unpack16(const uint4& w, float* x) {
  if constexpr (sizeof(TT) == 2) {
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
  } else {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
}

// Online (max, sum) update with one 16-byte vector of logits.
template <typename TT>
__device__ __forceinline__ void softmax_acc16(const uint4& w, float& m, float& s, float c) {
  constexpr int kEl = 16 / sizeof(TT);
  float x[kEl];
  unpack16<TT>(w, x);
  float vm = x[0];
#pragma unroll
  for (int k = 1; k < kEl; ++k) vm = fmaxf(vm, x[k]);
  if (vm > m) {
    s *= ex2((m - vm) * c);
    m = vm;
  }
  if (m != -INFINITY) {
    float a = 0.0f;
#pragma unroll
    for (int k = 0; k < kEl; ++k) a += ex2((x[k] - m) * c);
    s += a;
  }
}

// As softmax_acc16, with the sum kept as an unevaluated pair s + l: each
// vector's partial sum is added by Knuth's TwoSum, whose rounding error goes
// to l, so the row's sum does not lose the low bits of its many additions.
template <typename TT>
__device__ __forceinline__ void softmax_acc16_ff(const uint4& w, float& m, float& s, float& l,
                                                 float c) {
  constexpr int kEl = 16 / sizeof(TT);
  float x[kEl];
  unpack16<TT>(w, x);
  float vm = x[0];
#pragma unroll
  for (int k = 1; k < kEl; ++k) vm = fmaxf(vm, x[k]);
  if (vm > m) {
    const float f = ex2((m - vm) * c);
    s *= f;
    l *= f;
    m = vm;
  }
  if (m != -INFINITY) {
    float a = 0.0f;
#pragma unroll
    for (int k = 0; k < kEl; ++k) a += ex2((x[k] - m) * c);
    const float t = s + a;
    const float bp = t - s;
    l += (s - (t - bp)) + (a - bp);
    s = t;
  }
}

// Sweep-2 work on 4 consecutive vocabulary entries starting at v.  With kMask
// the entries below tau are outside the adjusted row (p = 0).
template <bool kHasQ, bool kRace, bool kMask>
__device__ __forceinline__ void sweep2_4(const float* l, const float4& q4, float M, float c,
                                         float invS, float tau, bool resid, uint64_t rkey,
                                         uint32_t v, float& beta, Race& best, int excl = -1) {
  const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
  float p[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) p[k] = ex2((l[k] - M) * c) * invS;
  if constexpr (kMask) {
#pragma unroll
    for (int k = 0; k < 4; ++k) p[k] = l[k] >= tau ? p[k] : 0.0f;
  }
  if constexpr (kHasQ)
    beta += (fminf(p[0], qv[0]) + fminf(p[1], qv[1])) + (fminf(p[2], qv[2]) + fminf(p[3], qv[3]));
  if constexpr (kRace) {
    float w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w[k] = (kHasQ && resid) ? fmaxf(p[k] - qv[k], 0.0f) : p[k];
      if (!kHasQ && (int)(v + k) == excl) w[k] = 0.0f;  // one-hot draft: residual is p without x
    }
    if constexpr (kMask) {
      // entries outside the adjusted row (and a zero residual) are no
      // candidates: a group without any skips its four hashes
      if (!((w[0] > 0.0f) | (w[1] > 0.0f) | (w[2] > 0.0f) | (w[3] > 0.0f))) return;
    }
    race_offer4(best, w, rkey, v);
  }
}

// Sweep 2 over vectors [lo, hi) of the row (elements [lo, hi) when the row is
// not 16-byte aligned).
template <typename TT, int NT, bool kHasQ, bool kRace, bool kMask = false>
__device__ __forceinline__ void sweep2(const TT* row, const float* qrow, int lo, int hi, bool vec,
                                       float M, float c, float invS, float tau, bool resid,
                                       uint64_t rkey, uint64_t pol, float& beta, Race& best,
                                       int excl = -1, bool sparse = false) {
  constexpr int kEl = 16 / sizeof(TT);
  // target vectors loaded per iteration: fewer where the race needs registers
  constexpr int U = kRace ? 2 : (sizeof(TT) == 2 ? 3 : 4);
  const int tid = threadIdx.x;
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (vec) {
    const uint4* rv = reinterpret_cast<const uint4*>(row);
    const uint4* qv = reinterpret_cast<const uint4*>(qrow);
    const int nv = hi;
    int j = lo + tid;
    int round = 0;
    // With the race the loop shuffles across the warp, so it runs only while
    // every lane of the warp (j = jw .. jw + 31) has a full step: j + lag is the
    // warp's last j.  What is left goes through the one-vector loop below.
    const int lag = kRace ? 31 - (tid & 31) : 0;
    if (kMask && !kRace && sparse) {
      // Adjusted rows that keep few entries: entries below tau have p' = 0, so
      // they add nothing to beta and are no race candidates.  A target vector
      // with no entry at or above tau is skipped whole, and its draft entries
      // are never loaded (a top-k row of V = 256000 keeps a few dozen entries:
      // nearly the whole draft row stays unread).  Skipping only drops
      // additions of zero, so the sums are the same as without the test.  Rows
      // that keep many entries, and the race (whose registers this loop's
      // would spill), take the loop below, whose draft loads do not wait for
      // the target vectors.
      constexpr int U2 = 2;
      for (; j + lag + (U2 - 1) * NT < nv; j += U2 * NT) {
        if constexpr (kRace) {
          if ((++round & 3) == 0) warp_race(best);
        }
        uint4 a[U2];
#pragma unroll
        for (int u = 0; u < U2; ++u) a[u] = ldg_hint(rv + j + u * NT, pol);
        bool keep[U2];
#pragma unroll
        for (int u = 0; u < U2; ++u) {
          float x[kEl];
          unpack16<TT>(a[u], x);
          keep[u] = false;
#pragma unroll
          for (int e = 0; e < kEl; ++e) keep[u] |= x[e] >= tau;
        }
        uint4 b[U2][kEl / 4];
        if constexpr (kHasQ) {
#pragma unroll
          for (int u = 0; u < U2; ++u)
            if (keep[u]) {
#pragma unroll
              for (int h = 0; h < kEl / 4; ++h) b[u][h] = ldg_hint(qv + (j + u * NT) * (kEl / 4) + h, pol);
            }
        }
#pragma unroll
        for (int u = 0; u < U2; ++u) {
          if (!keep[u]) continue;
          float x[kEl];
          unpack16<TT>(a[u], x);
#pragma unroll
          for (int h = 0; h < kEl / 4; ++h) {
            float4 q4 = zero4;
            if constexpr (kHasQ) q4 = *reinterpret_cast<const float4*>(&b[u][h]);
            sweep2_4<kHasQ, kRace, kMask>(x + 4 * h, q4, M, c, invS, tau, resid, rkey,
                                          (uint32_t)((j + u * NT) * kEl + 4 * h), beta, best, excl);
          }
        }
      }
      for (; j < nv; j += NT) {
        float x[kEl];
        unpack16<TT>(ldg_hint(rv + j, pol), x);
        bool keep = false;
#pragma unroll
        for (int e = 0; e < kEl; ++e) keep |= x[e] >= tau;
        if (!keep) continue;
#pragma unroll
        for (int h = 0; h < kEl / 4; ++h) {
          float4 q4 = zero4;
          if constexpr (kHasQ) {
            uint4 w = ldg_hint(qv + j * (kEl / 4) + h, pol);
            q4 = *reinterpret_cast<const float4*>(&w);
          }
          sweep2_4<kHasQ, kRace, kMask>(x + 4 * h, q4, M, c, invS, tau, resid, rkey,
                                        (uint32_t)(j * kEl + 4 * h), beta, best, excl);
        }
      }
      return;
    }
    for (; j + lag + (U - 1) * NT < nv; j += U * NT) {
      if constexpr (kRace) {
        // every few rounds each lane takes the warp's best so far, so the
        // pruning bound tightens early (any entry already offered is a valid best)
        if ((++round & 3) == 0) warp_race(best);
      }
      uint4 a[U];
      uint4 b[U][kEl / 4];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        a[u] = ldg_hint(rv + j + u * NT, pol);
        if constexpr (kHasQ) {
#pragma unroll
          for (int h = 0; h < kEl / 4; ++h) b[u][h] = ldg_hint(qv + (j + u * NT) * (kEl / 4) + h, pol);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float x[kEl];
        unpack16<TT>(a[u], x);
#pragma unroll
        for (int h = 0; h < kEl / 4; ++h) {
          float4 q4 = zero4;
          if constexpr (kHasQ) q4 = *reinterpret_cast<const float4*>(&b[u][h]);
          sweep2_4<kHasQ, kRace, kMask>(x + 4 * h, q4, M, c, invS, tau, resid, rkey,
                                        (uint32_t)((j + u * NT) * kEl + 4 * h), beta, best, excl);
        }
      }
    }
    for (; j < nv; j += NT) {
      float x[kEl];
      unpack16<TT>(ldg_hint(rv + j, pol), x);
#pragma unroll
      for (int h = 0; h < kEl / 4; ++h) {
        float4 q4 = zero4;
        if constexpr (kHasQ) {
          uint4 w = ldg_hint(qv + j * (kEl / 4) + h, pol);
          q4 = *reinterpret_cast<const float4*>(&w);
        }
        sweep2_4<kHasQ, kRace, kMask>(x + 4 * h, q4, M, c, invS, tau, resid, rkey,
                                      (uint32_t)(j * kEl + 4 * h), beta, best, excl);
      }
    }
  } else {
    for (int v = lo + tid; v < hi; v += NT) {
      const float xv = load_logit(row + v);
      float p = ex2((xv - M) * c) * invS;
      if constexpr (kMask) p = xv >= tau ? p : 0.0f;
      float qv = 0.0f;
      if constexpr (kHasQ) {
        qv = __ldg(qrow + v);
        beta += fminf(p, qv);
      }
      if constexpr (kRace)
        race_offer(best, (kHasQ && resid) ? fmaxf(p - qv, 0.0f) : (v == excl ? 0.0f : p), rkey,
                   (uint32_t)v);
    }
  }
}

// Sweep 2 of an adjusted row whose kept entries are all in its candidate list
// (index and value of every entry at or above the counting pass's bound): beta
// and the race over the listed entries at or above tau, with the same per-entry
// arithmetic as sweep2 (every other entry has p' = 0: nothing to beta, no race
// candidate; the race's winner does not depend on the order of the offers).
template <int NT, bool kHasQ, bool kRace>
__device__ __forceinline__ void sweep2_list(const uint2* cand, int n, const float* qrow, float M,
                                            float c, float invS, float tau, bool resid,
                                            uint64_t rkey, float& beta, Race& best, int excl) {
  for (int i = threadIdx.x; i < n; i += NT) {
    const uint2 e = cand[i];
    const float x = __uint_as_float(e.y);
    if (!(x >= tau)) continue;
    const float p = ex2((x - M) * c) * invS;
    float q = 0.0f;
    if constexpr (kHasQ) {
      q = __ldg(qrow + e.x);
      beta += fminf(p, q);
    }
    if constexpr (kRace) {
      const float w = (kHasQ && resid) ? fmaxf(p - q, 0.0f) : ((int)e.x == excl ? 0.0f : p);
      race_offer(best, w, rkey, e.x);
    }
  }
}

// Sweep 1 over vectors [lo, hi) (elements when not aligned): per-thread online
// (max, sum) in two interleaved accumulators, merged on return.
template <typename TT, int NT>
__device__ __forceinline__ void sweep1(const TT* row, int lo, int hi, bool vec, float c,
                                       uint64_t pol, float& m, float& s) {
  float m0 = -INFINITY, s0 = 0.0f, m1 = -INFINITY, s1 = 0.0f;
  const int tid = threadIdx.x;
  if (vec) {
    const uint4* rv = reinterpret_cast<const uint4*>(row);
    int j = lo + tid;
    for (; j + 7 * NT < hi; j += 8 * NT) {   // 8 vectors (128 B) in flight per thread
      uint4 a[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = ldg_hint(rv + j + u * NT, pol);
#pragma unroll
      for (int u = 0; u < 8; u += 2) {
        softmax_acc16<TT>(a[u], m0, s0, c);
        softmax_acc16<TT>(a[u + 1], m1, s1, c);
      }
    }
    for (; j < hi; j += NT) softmax_acc16<TT>(ldg_hint(rv + j, pol), m0, s0, c);
  } else {
    for (int v = lo + tid; v < hi; v += NT) {
      const float xv = load_logit(row + v);
      if (xv > m0) {
        s0 *= ex2((m0 - xv) * c);
        m0 = xv;
      }
      if (m0 != -INFINITY) s0 += ex2((xv - m0) * c);
    }
  }
  softmax_merge(m0, s0, m1, s1, c);
  m = m0;
  s = s0;
}

// Sweep 1 of the adjusted kernel: as sweep1, with the per-thread sum carried
// as s + l (softmax_acc16_ff); the two accumulators are merged with the
// products' and the addition's rounding errors moved to l.
template <typename TT, int NT>
__device__ __forceinline__ void sweep1_ff(const TT* row, int hi, bool vec, float c, uint64_t pol,
                                          float& m, float& s, float& l) {
  float m0 = -INFINITY, s0 = 0.0f, l0 = 0.0f, m1 = -INFINITY, s1 = 0.0f, l1 = 0.0f;
  const int tid = threadIdx.x;
  if (vec) {
    const uint4* rv = reinterpret_cast<const uint4*>(row);
    int j = tid;
    for (; j + 7 * NT < hi; j += 8 * NT) {
      uint4 a[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = ldg_hint(rv + j + u * NT, pol);
#pragma unroll
      for (int u = 0; u < 8; u += 2) {
        softmax_acc16_ff<TT>(a[u], m0, s0, l0, c);
        softmax_acc16_ff<TT>(a[u + 1], m1, s1, l1, c);
      }
    }
    for (; j < hi; j += NT) softmax_acc16_ff<TT>(ldg_hint(rv + j, pol), m0, s0, l0, c);
  } else {
    for (int v = tid; v < hi; v += NT) {
      const float xv = load_logit(row + v);
      if (xv > m0) {
        const float f = ex2((m0 - xv) * c);
        s0 *= f;
        l0 *= f;
        m0 = xv;
      }
      if (m0 != -INFINITY) {
        const float a = ex2((xv - m0) * c);
        const float t = s0 + a;
        const float bp = t - s0;
        l0 += (s0 - (t - bp)) + (a - bp);
        s0 = t;
      }
    }
  }
  const float mn = fmaxf(m0, m1);
  if (mn == -INFINITY) {
    m = mn;
    s = 0.0f;
    l = 0.0f;
    return;
  }
  const float f0 = ex2((m0 - mn) * c), f1 = ex2((m1 - mn) * c);
  const float a = s0 * f0, b = s1 * f1;
  const float t = a + b;
  const float bp = t - a;
  m = mn;
  s = t;
  l = (l0 * f0 + l1 * f1) + ((a - (t - bp)) + (b - bp)) + (fmaf(s0, f0, -a) + fmaf(s1, f1, -b));
}

// ---------------------------------------------------------------------------
// Top-k / top-p adjusted target rows (the vllbc page's Section 2.2 note: top-k
// and top-p fold into the adjusted p before the same rejection test).
//
// Kept set of a row, with masses e(v) of the logits:
//   top-k (1 <= k < V): v with fewer than k logits above l_v (ties at the k-th
//                       largest logit all stay);
//   top-p (P < 1):      v with A(v) = 0 or A(v) < P * S_k, A(v) the mass of the
//                       logits above l_v and S_k the mass kept by top-k.
// Both are a threshold on the logit: the kept set is {v : l_v >= tau}.  tau is
// found by a selection over the row while it is still in L2:
//   1. an estimate: a histogram of one 16-byte vector in 16, binned by
//      z = (M - l) c (64 bins per unit of z), gives the z by which the edge
//      should have been passed; the cut Zc is set a margin beyond it;
//   2. the entries with z < Zc go into 2048 bins of width 2^-a (a as fine as
//      the cut allows) with their count, mass and smallest / largest logit
//      key; every other entry is only counted (and its mass summed, when the
//      top-p bound needs the whole row) in registers;
//   3. the bin where the criterion is met either holds one logit value (done)
//      or is split by its keys into 1024 sub-bins, again until one value is
//      left.
// When the edge lies beyond Zc (or in a row holding -inf or NaN at the edge)
// step 2 runs again with 64 bins per unit and a last bin that takes the rest.
// bf16 rows whose entries above the cut take at most 2048 values (the common
// case: the values between the cut and the max span a few octaves of 128
// bf16 values each) replace steps 2 and 3 by one pass with a bin per value:
// one 32-bit count per entry, the bin's mass its count times the value's mass
// (adj_run_keys); the top-p bound without top-k then takes the row's whole
// mass from sweep 1, summed with error compensation and added up as integers
// of the same scale.
// Counts are exact; masses are integers (pow2_neg(z) scaled by 2^F with
// V 2^F <= 2^62), so the shared-memory histograms add up the same way in any
// order, the result does not depend on thread timing, and the top-p test
// (double)A < (double)P * (double)S_k sees the numbers a CPU restatement sees.
// ---------------------------------------------------------------------------
constexpr int kAdjBins1 = 2048;
constexpr int kAdjBins2 = 1024;
constexpr int kAdjSample = 16;       // the estimate reads one vector (or element) in 16
constexpr int kAdjMaxKeyLevels = 4;  // 1024^4 > 2^32: key levels always end on one value
constexpr int kAdjCand = 2048;       // candidate list of a top-k row (index, value)

// Selection statistics (specdec_set_adjust_counters): adjusted rows, rows whose
// sample put the edge in the last bin, rows whose edge lay past the cut,
// key-refinement passes, rows left without a threshold, rows resolved on
// bins of one bf16 value each.
enum AdjCounter {
  kAdjRows = 0, kAdjTail, kAdjMiss, kAdjKeyPass, kAdjNone, kAdjExact, kAdjCounters = 8
};
__device__ __forceinline__ void adj_count(unsigned long long* ctr, int i) {
  if (ctr && threadIdx.x == 0) atomicAdd(ctr + i, 1ull);
}

struct AdjShared {
  uint32_t cnt1[kAdjBins1];
  unsigned long long mass1[kAdjBins1];
  uint32_t kmin1[kAdjBins1];
  uint32_t kmax1[kAdjBins1];
  uint32_t cnt2[kAdjBins2];
  unsigned long long mass2[kAdjBins2];
  uint32_t kmin2[kAdjBins2];
  uint32_t kmax2[kAdjBins2];
  uint32_t wcnt[32];
  unsigned long long wmass[32];
  int sel;
  uint32_t ex_cnt;
  unsigned long long ex_mass;
  uint2 cand[kAdjCand];  // (index, logit bits) of the entries a counting pass saw
  int ncand;
};

// Mass of an entry for the selection: 2^-z on a float32 definition that a CPU
// implementation can reproduce bit for bit, so that the top-p edge (a decision
// floating point takes) comes out the same on both: 0 for z >= 64 (or NaN);
// otherwise 2^-f * 2^-k with k = floor(z), f = z - k, and 2^-f the Taylor
// series of degree 8, coefficients (-ln 2)^n / n! rounded to float32, by
// Horner's rule with fused multiply-adds.  Within 4e-7 of 2^-z.
__device__ __forceinline__ float pow2_neg(float z) {
  if (!(z < 64.0f)) return 0.0f;
  const int k = (int)z;
  const float f = z - (float)k;
  float q = 1.3215486790144305e-06f;
  q = __fmaf_rn(q, f, -1.5252733804059838e-05f);
  q = __fmaf_rn(q, f, 0.00015403530393381606f);
  q = __fmaf_rn(q, f, -0.0013333558146428441f);
  q = __fmaf_rn(q, f, 0.009618129107628477f);
  q = __fmaf_rn(q, f, -0.055504108664821576f);
  q = __fmaf_rn(q, f, 0.2402265069591007f);
  q = __fmaf_rn(q, f, -0.6931471805599453f);
  q = __fmaf_rn(q, f, 1.0f);
  return q * __int_as_float((127 - k) << 23);  // exact: q >= 1/2, k <= 63
}

// Integer masses of a row of V entries are pow2_neg(z) scaled by 2^F,
// F = 62 - ceil(log2 V), so that a whole row's masses sum below 2^62; each is
// rounded to the nearest integer (ties to even).
__device__ __forceinline__ int adj_mass_shift(int V) {
  const int lg = V > 1 ? 32 - __clz(V - 1) : 0;
  return 62 - lg;
}
__device__ __forceinline__ float adj_mass_scale(int F) { return __int_as_float((127 + F) << 23); }
__device__ __forceinline__ unsigned long long adj_mass(float z, float fscale) {
  return __float2ull_rn(pow2_neg(z) * fscale);
}

// Order-preserving key of a logit (-0.0 folded into +0.0).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// 16-bit order key of a bf16 value held as a float (the upper half of its
// order key: distinct bf16 values get distinct, ordered keys), and back.
__device__ __forceinline__ uint32_t key16(float x) { return order_key(x) >> 16; }
__device__ __forceinline__ float key16_value(uint32_t k) {
  return key_value((k << 16) | ((k & 0x8000u) ? 0u : 0xFFFFu));
}

// Level-1 geometry: bins of width 1/scale in z (scale a power of two).  With
// catch_all the last bin also takes every z past the grid, NaN included;
// otherwise only z < cut is binned and the rest is "far".
// With lo > 0 (top-p alone, when the sample pins the edge down) the bins cover
// only the window [lo, cut): entries with z < lo lie above the edge, so only
// their count and mass are needed, and those are summed in registers.
struct AdjGrid {
  float scale;
  float cut;
  bool catch_all;
  float lo;
};

__device__ __forceinline__ int adj_bin1(float z, const AdjGrid& g) {
  if (g.catch_all) {
    const float y = z * g.scale;
    return y < (float)(kAdjBins1 - 1) ? (int)y : kAdjBins1 - 1;
  }
  if (!(z < g.cut)) return -1;
  if (z < g.lo) return -2;
  const int b = (int)((z - g.lo) * g.scale);  // monotone in z, so in the logit
  return b < kAdjBins1 ? b : kAdjBins1 - 1;  // the cut lies inside the grid; guard only
}

// Visits every entry of the row (or, with kSampled, one 16-byte vector in 16,
// one element in 16 on unaligned rows) through f(x), and calls g() after each
// vector (each element on unaligned rows).
struct AdjNoFlush {
  __device__ __forceinline__ void operator()() const {}
};
template <typename TT, int NT, bool kSampled, typename Fn, typename Gn = AdjNoFlush>
__device__ __forceinline__ void adj_visit(const TT* row, int V, bool vec, uint64_t pol, Fn&& f,
                                          Gn&& g = Gn()) {
  constexpr int kEl = 16 / sizeof(TT);
  constexpr int kStep = kSampled ? kAdjSample : 1;
  const int tid = threadIdx.x;
  if (vec) {
    // one copy of the per-vector body (f is inlined kEl times, not 3 kEl): the
    // next vector's load is issued before the current one is processed
    const uint4* rv = reinterpret_cast<const uint4*>(row);
    const int nv = V / kEl;
    int j = tid * kStep;
    if (j < nv) {
      uint4 cur = ldg_hint(rv + j, pol);
#pragma unroll 1
      for (;;) {
        const int jn = j + NT * kStep;
        uint4 nxt = cur;
        if (jn < nv) nxt = ldg_hint(rv + jn, pol);
        float x[kEl];
        unpack16<TT>(cur, x);
#pragma unroll
        for (int e = 0; e < kEl; ++e) f(x[e]);
        g();
        if (jn >= nv) break;
        cur = nxt;
        j = jn;
      }
    }
  } else {
    for (int v = tid * kStep; v < V; v += NT * kStep) {
      f(load_logit(row + v));
      g();
    }
  }
}

// Visits every entry of the row through f(x, n, v), a vector at a time: n = kEl
// values of one 16-byte vector, or n = 1 on unaligned rows; v = the index of x[0].
template <typename TT, int NT, typename Fn>
__device__ __forceinline__ void adj_visit_vec(const TT* row, int V, bool vec, uint64_t pol, Fn&& f) {
  constexpr int kEl = 16 / sizeof(TT);
  const int tid = threadIdx.x;
  if (vec) {
    const uint4* rv = reinterpret_cast<const uint4*>(row);
    const int nv = V / kEl;
    int j = tid;
    if (j < nv) {
      uint4 cur = ldg_hint(rv + j, pol);
#pragma unroll 1
      for (;;) {
        const int jn = j + NT;
        uint4 nxt = cur;
        if (jn < nv) nxt = ldg_hint(rv + jn, pol);
        float x[kEl];
        unpack16<TT>(cur, x);
        f(x, kEl, j * kEl);
        if (jn >= nv) break;
        cur = nxt;
        j = jn;
      }
    }
  } else {
    for (int v = tid; v < V; v += NT) {
      float x[kEl];
      x[0] = load_logit(row + v);
      f(x, 1, v);
    }
  }
}

// As adj_visit_vec, with four vectors loaded before any is processed (the
// counting pass of adj_run_keys reads rows that L2 has mostly let go, so it
// needs more loads in flight than the passes served from L2).
template <typename TT, int NT, typename Fn>
__device__ __forceinline__ void adj_visit_vec4(const TT* row, int V, bool vec, uint64_t pol, Fn&& f) {
  constexpr int kEl = 16 / sizeof(TT);
  const int tid = threadIdx.x;
  if (vec) {
    const uint4* rv = reinterpret_cast<const uint4*>(row);
    const int nv = V / kEl;
    int j = tid;
    for (; j + 3 * NT < nv; j += 4 * NT) {
      uint4 a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = ldg_hint(rv + j + u * NT, pol);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float x[kEl];
        unpack16<TT>(a[u], x);
        f(x, kEl, (j + u * NT) * kEl);
      }
    }
    for (; j < nv; j += NT) {
      float x[kEl];
      unpack16<TT>(ldg_hint(rv + j, pol), x);
      f(x, kEl, j * kEl);
    }
  } else {
    for (int v = tid; v < V; v += NT) {
      float x[kEl];
      x[0] = load_logit(row + v);
      f(x, 1, v);
    }
  }
}

// First bin j of [0, n) (bins run from the largest logits down) at which
//   by count: the running count through j reaches `need`;
//   by mass:  cnt[j] > 0 and above + the running mass through j >= bound.
// Leaves j in A.sel (n when no bin qualifies) and the count and mass of the
// bins before it in A.ex_cnt / A.ex_mass.  Block-wide; ends on a barrier.
template <int NT>
__device__ __forceinline__ void adj_select(const uint32_t* cnt, const unsigned long long* mass,
                                           int n, bool by_mass, uint32_t need, double bound,
                                           unsigned long long above, AdjShared& A) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = n / NT;
  const int j0 = tid * per;
  uint32_t lc = 0;
  unsigned long long lm = 0;
  for (int q = 0; q < per; ++q) {
    lc += cnt[j0 + q];
    lm += mass[j0 + q];
  }
  uint32_t ic = lc;
  unsigned long long im = lm;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t c2 = __shfl_up_sync(0xFFFFFFFFu, ic, o);
    const unsigned long long m2 = __shfl_up_sync(0xFFFFFFFFu, im, o);
    if (lane >= o) {
      ic += c2;
      im += m2;
    }
  }
  if (lane == 31) {
    A.wcnt[warp] = ic;
    A.wmass[warp] = im;
  }
  if (tid == 0) A.sel = n;
  __syncthreads();
  uint32_t ec = ic - lc;
  unsigned long long em = im - lm;
  for (int w = 0; w < warp; ++w) {
    ec += A.wcnt[w];
    em += A.wmass[w];
  }
  uint32_t rc = ec;
  unsigned long long rm = em;
  int found = -1;
  for (int q = 0; q < per; ++q) {
    const int j = j0 + q;
    rc += cnt[j];
    rm += mass[j];
    const bool ok = by_mass ? (cnt[j] > 0 && (double)(above + rm) >= bound) : (rc >= need);
    if (ok) {
      found = j;
      break;
    }
  }
  if (found >= 0) atomicMin(&A.sel, found);
  __syncthreads();
  const int sel = A.sel;
  if (sel < n && sel >= j0 && sel < j0 + per) {
    for (int j = j0; j < sel; ++j) {
      ec += cnt[j];
      em += mass[j];
    }
    A.ex_cnt = ec;
    A.ex_mass = em;
  }
  __syncthreads();
}

// Sum of one value over the block (deterministic).  Ends on a barrier.
template <int NT>
__device__ __forceinline__ unsigned long long adj_block_sum(unsigned long long x, AdjShared& A) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  if (lane == 0) A.wmass[warp] = x;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < NT / 32; ++w) t += A.wmass[w];
  __syncthreads();
  return t;
}

// Splits the chosen bin, whose entries are exactly those with keys in
// [lo, hi] (z is monotone in the logit), by keys into 1024 sub-bins (sub-bin 0
// holds the largest keys) until the criterion (see adj_select) is met on a
// single logit value.  above_c / above_m: count and mass of every entry with a
// key above hi; m_sel: the chosen bin's mass.  Returns the value's key and the
// mass of every entry whose key is >= it; false when no sub-bin qualifies.
template <typename TT, int NT>
__device__ bool adj_refine(const TT* row, int V, bool vec, float M, float c, float fscale,
                           bool by_mass, uint32_t need, double bound, uint32_t above_c,
                           unsigned long long above_m, uint32_t lo, uint32_t hi,
                           unsigned long long m_sel, uint32_t c_sel, uint64_t pol, AdjShared& A,
                           uint32_t& key, unsigned long long& kept, uint32_t& kept_cnt,
                           unsigned long long* ctr) {
  const int tid = threadIdx.x;
  if (lo > hi) return false;
  for (int level = 0; level <= kAdjMaxKeyLevels; ++level) {
    if (lo == hi) {
      key = lo;
      kept = above_m + m_sel;
      kept_cnt = above_c + c_sel;
      return true;
    }
    const uint32_t w = (uint32_t)(((unsigned long long)hi - lo + kAdjBins2) / kAdjBins2);
    adj_count(ctr, kAdjKeyPass);
    for (int j = tid; j < kAdjBins2; j += NT) {
      A.cnt2[j] = 0u;
      A.mass2[j] = 0ull;
      A.kmin2[j] = 0xFFFFFFFFu;
      A.kmax2[j] = 0u;
    }
    __syncthreads();
    adj_visit<TT, NT, false>(row, V, vec, pol, [&](float x) {
      const uint32_t k = order_key(x);
      if (k < lo || k > hi) return;
      const uint32_t s = (hi - k) / w;
      if (s >= (uint32_t)kAdjBins2) return;  // cannot happen; guard only
      atomicAdd(&A.cnt2[s], 1u);
      atomicAdd(&A.mass2[s], adj_mass((M - x) * c, fscale));
      atomicMin(&A.kmin2[s], k);
      atomicMax(&A.kmax2[s], k);
    });
    __syncthreads();
    adj_select<NT>(A.cnt2, A.mass2, kAdjBins2, by_mass, need - above_c, bound, above_m, A);
    const int s = A.sel;
    if (s < kAdjBins2) {
      above_c += A.ex_cnt;
      above_m += A.ex_mass;
      lo = A.kmin2[s];
      hi = A.kmax2[s];
      m_sel = A.mass2[s];
      c_sel = A.cnt2[s];
    }
    __syncthreads();
    if (s >= kAdjBins2 || lo > hi) return false;
  }
  return false;
}

// Every entry with z < cut (all of them with catch_all) goes into the level-1
// bins with its count, mass and key range (the others are only counted, and
// their mass summed when the top-p bound needs the whole row); then the top-k
// and top-p edges.  Returns false when an edge lies past the grid (only
// possible without catch_all) or the row holds NaN.
template <typename TT, int NT>
__device__ bool adj_run(const TT* row, int V, bool vec, float M, float c, float fscale, int top_k,
                        float top_p, bool use_k, bool use_p, const AdjGrid& g, uint64_t pol,
                        AdjShared& A, uint32_t& key, unsigned long long& kept,
                        uint32_t& kept_cnt, unsigned long long* ctr) {
  const int tid = threadIdx.x;
  for (int j = tid; j < kAdjBins1; j += NT) {
    A.cnt1[j] = 0u;
    A.mass1[j] = 0ull;
    A.kmin1[j] = 0xFFFFFFFFu;
    A.kmax1[j] = 0u;
  }
  __syncthreads();
  // The far entries' mass matters only for a top-p bound over the whole row.
  // Each far entry's 2^-z comes from the special-function unit (relative error
  // below 2^-22) and is summed in float32 over one vector (at most 8 terms),
  // then added as an integer: the sum is within 1e-6 relative of the exact one,
  // which decides the edge the same way everywhere outside the 1e-5 band the
  // oracle reports.
  // Entries above a window (z < g.lo) are counted and their masses summed the
  // same way, apart from the far ones.
  // Each vector is classified first; the atomics of its window entries follow
  // in one loop, so a warp issues them about as often as its busiest lane has
  // window entries in the vector, not once per element position that any lane
  // has one.
  constexpr int kEl = 16 / sizeof(TT);
  const bool far_mass = use_p && !use_k;
  const bool windowed = g.lo > 0.0f;
  unsigned long long fm = 0, um = 0;
  uint32_t uc = 0;
  adj_visit_vec<TT, NT>(row, V, vec, pol, [&](const float* x, int n, int) {
    uint32_t wm = 0;
    float fv = 0.0f, uv = 0.0f;
#pragma unroll
    for (int e = 0; e < kEl; ++e) {
      if (e >= n) break;
      const float z = (M - x[e]) * c;
      const int b = adj_bin1(z, g);
      if (b == -2) {
        ++uc;
        uv += ex2(-z);
      } else if (b < 0) {
        if (far_mass && z < 64.0f) fv += ex2(-z);  // NaN and z >= 64 add nothing
      } else {
        wm |= 1u << e;
      }
    }
    if (far_mass) fm += __float2ull_rn(fv * fscale);
    if (windowed) um += __float2ull_rn(uv * fscale);
    while (wm) {
      const int e = __ffs(wm) - 1;
      wm &= wm - 1;
      float xe = x[0];
#pragma unroll
      for (int k = 1; k < kEl; ++k) xe = (e == k) ? x[k] : xe;
      const float z = (M - xe) * c;
      const int b = adj_bin1(z, g);
      const uint32_t k = order_key(xe);
      atomicAdd(&A.cnt1[b], 1u);
      atomicAdd(&A.mass1[b], adj_mass(z, fscale));
      atomicMin(&A.kmin1[b], k);
      atomicMax(&A.kmax1[b], k);
    }
  });
  __syncthreads();
  unsigned long long tm = fm + um;
  for (int j = tid; j < kAdjBins1; j += NT) tm += A.mass1[j];
  kept = adj_block_sum<NT>(tm, A);
  const unsigned long long above_m = windowed ? adj_block_sum<NT>(um, A) : 0ull;
  const uint32_t above_c = windowed ? (uint32_t)adj_block_sum<NT>(uc, A) : 0u;
  key = 0u;  // below every logit
  for (int pass = 0; pass < 2; ++pass) {
    const bool by_mass = pass == 1;
    if (by_mass ? !use_p : !use_k) continue;
    const double bound =
        by_mass ? (top_p > 0.0f ? (double)top_p : 0.0) * (double)kept : 0.0;
    // the edge must lie in the window: the entries above it must not reach
    // the bound (the first group, A = 0, is kept regardless)
    if (above_c > 0 && (by_mass ? (double)above_m >= bound : above_c >= (uint32_t)top_k))
      return false;
    adj_select<NT>(A.cnt1, A.mass1, kAdjBins1, by_mass, (uint32_t)top_k - above_c, bound, above_m,
                   A);
    const int j1 = A.sel;
    uint32_t ac = 0, lo = 1, hi = 0, cs = 0;
    unsigned long long am = 0, ms = 0;
    if (j1 < kAdjBins1) {
      ac = A.ex_cnt + above_c;
      am = A.ex_mass + above_m;
      lo = A.kmin1[j1];
      hi = A.kmax1[j1];
      ms = A.mass1[j1];
      cs = A.cnt1[j1];
    }
    __syncthreads();
    if (!adj_refine<TT, NT>(row, V, vec, M, c, fscale, by_mass, (uint32_t)top_k, bound, ac, am,
                            lo, hi, ms, cs, pol, A, key, kept, kept_cnt, ctr))
      return false;
  }
  return true;
}

// bf16 rows whose entries at or above x_lo take at most 2048 values
// (key16(M) - key16(x_lo) < 2048): one pass counts the entries of each value in
// bin j = key16(M) - key16(x) (bin 0 holds the max).  A bin holds one value, so
// its mass is its count times that value's integer mass (the sum of the
// per-entry masses), no key refinement follows, and an entry costs one 32-bit
// shared-memory atomic.  Entries below x_lo (and NaN) are not counted: the top-k
// edge needs only the counts above it, and the top-p bound is P times the
// top-k set's mass, or, without top-k, P times s_all, the row's whole mass on
// the same integer scale.  False when an edge lies below x_lo.
// With record, the counted entries' indices and values also go to A.cand;
// ncand is then their number (every entry at or above x_lo, so every kept
// one), or -1 when they did not fit (and always -1 without record).
template <int NT, bool kDeep>
__device__ bool adj_run_keys(const __nv_bfloat16* row, int V, bool vec, float M, float c,
                             float fscale, int top_k, float top_p, bool use_k, bool use_p,
                             unsigned long long s_all, float x_lo, bool record, uint64_t pol,
                             AdjShared& A, uint32_t& key, unsigned long long& kept,
                             uint32_t& kept_cnt, int& ncand) {
  const int tid = threadIdx.x;
  const uint32_t ktop = key16(M);
  for (int j = tid; j < kAdjBins1; j += NT) A.cnt1[j] = 0u;
  if (tid == 0) A.ncand = 0;
  __syncthreads();
  auto count = [&](const float* x, int n, int v0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (e < n && x[e] >= x_lo) {
        // x <= M, and x >= x_lo bounds the key from below: j < 2048 (guard only)
        const uint32_t j = ktop - key16(x[e]);
        atomicAdd(&A.cnt1[j < (uint32_t)kAdjBins1 ? j : kAdjBins1 - 1], 1u);
        if (record) {
          const int pos = atomicAdd(&A.ncand, 1);
          if (pos < kAdjCand) A.cand[pos] = make_uint2((uint32_t)(v0 + e), __float_as_uint(x[e]));
        }
      }
    }
  };
  // rows bounded by the threads' maxima count few entries and need the row
  // back from DRAM fast (four vectors in flight); the others count many and
  // keep the smaller loop
  if constexpr (kDeep)
    adj_visit_vec4<__nv_bfloat16, NT>(row, V, vec, pol, count);
  else
    adj_visit_vec<__nv_bfloat16, NT>(row, V, vec, pol, count);
  __syncthreads();
  ncand = (record && A.ncand <= kAdjCand) ? A.ncand : -1;
  for (int j = tid; j < kAdjBins1; j += NT) {
    const uint32_t n = A.cnt1[j];
    A.mass1[j] =
        n ? (unsigned long long)n * adj_mass((M - key16_value(ktop - j)) * c, fscale) : 0ull;
  }
  __syncthreads();
  int j = kAdjBins1;
  uint32_t kc = 0u;
  unsigned long long km = 0ull;
  for (int pass = 0; pass < 2; ++pass) {
    const bool by_mass = pass == 1;
    if (by_mass ? !use_p : !use_k) continue;
    const double base = use_k ? (double)km : (double)s_all;
    const double bound = by_mass ? (top_p > 0.0f ? (double)top_p : 0.0) * base : 0.0;
    adj_select<NT>(A.cnt1, A.mass1, kAdjBins1, by_mass, (uint32_t)top_k, bound, 0ull, A);
    j = A.sel;
    if (j < kAdjBins1) {
      kc = A.ex_cnt + A.cnt1[j];
      km = A.ex_mass + A.mass1[j];
    }
    __syncthreads();
    if (j >= kAdjBins1) return false;
  }
  key = order_key(key16_value(ktop - j));
  kept = km;
  kept_cnt = kc;
  return true;
}

// The cut for the level-1 histogram from a sample of the row: the z (64 bins
// per unit) by which the sample passes 1.5 times its share of the top-k count,
// or, for top-p alone, where the sample's tail beyond z (16 times its mass)
// falls to (1 - P) S, S the row's softmax sum (the tail is made of many light
// entries, so its estimate is steadier than one of the few heavy ones at the
// top); plus a margin.  With both, the top-p edge lies inside the top-k set.
// False when the sample puts the edge in the last bin.
template <typename TT, int NT>
__device__ bool adj_estimate(const TT* row, int V, bool vec, float M, float c, float S,
                             int top_k, float top_p, bool use_k, bool use_p, uint64_t pol,
                             AdjShared& A, AdjGrid& g, AdjGrid& gw) {
  const int tid = threadIdx.x;
  const AdjGrid coarse{64.0f, 0.0f, true};
  for (int j = tid; j < kAdjBins1; j += NT) A.cnt1[j] = 0u;
  __syncthreads();
  adj_visit<TT, NT, true>(row, V, vec, pol, [&](float x) {
    atomicAdd(&A.cnt1[adj_bin1((M - x) * c, coarse)], 1u);
  });
  __syncthreads();
  // mass of a bin taken at its centre, in units of 2^-32
  unsigned long long tm = 0;
  for (int j = tid; j < kAdjBins1; j += NT) {
    A.mass1[j] = (unsigned long long)A.cnt1[j] *
                 (unsigned long long)exp2f(32.0f - ((float)j + 0.5f) * (1.0f / 64.0f));
    tm += A.mass1[j];
  }
  __syncthreads();
  const unsigned long long s_sample = adj_block_sum<NT>(tm, A);
  if (use_k) {
    // aim past the sample's share of k (a sample that happens to hold more
    // than its share of the top-k set stays inside)
    const int share = (top_k + kAdjSample - 1) / kAdjSample;
    adj_select<NT>(A.cnt1, A.mass1, kAdjBins1, false, (uint32_t)(share + share / 2 + 2), 0.0,
                   0ull, A);
  } else {
    const double p = top_p > 0.0f ? (double)top_p : 0.0;
    const double tail = (1.0 - p) * (double)S * 4294967296.0 / (double)kAdjSample;
    adj_select<NT>(A.cnt1, A.mass1, kAdjBins1, true, 0u, (double)s_sample - tail, 0ull, A);
  }
  const int j = A.sel;
  __syncthreads();
  if (j >= kAdjBins1 - 1) return false;
  const float z_est = (float)(j + 1) * (1.0f / 64.0f);
  // finest power-of-two bin width whose 2048 bins still cover [lo, cut)
  auto fit = [](AdjGrid& q) {
    const float span = q.cut - q.lo;
    int a = 6;
    while (a < 24 && (float)kAdjBins1 / (float)(1 << (a + 1)) >= span) ++a;
    while (a > -8 && (float)kAdjBins1 * exp2f((float)-a) < span) --a;
    q.scale = exp2f((float)a);
    q.catch_all = false;
  };
  g.cut = 1.0625f * z_est + 0.5f;
  g.lo = 0.0f;
  fit(g);
  gw = g;
  if (!use_k && top_p >= 0.7f) {
    // The sample's tail mass pins a top-p edge with P >= 0.7 down to a few
    // hundredths of a unit of z (the tail holds many light entries): the
    // window grid bins only a band around it.
    const float m = 0.3125f + 0.03125f * z_est;
    gw.cut = z_est + m;
    gw.lo = fmaxf(z_est - m, 0.0f);
    fit(gw);
  }
  return true;
}

// Threshold tau (keep l >= tau), kept mass S and number of kept entries of an
// adjusted row whose max is M; S holds the row's softmax sum on entry.
// Block-wide (every thread of the block calls it with the same arguments).
// Returns false, leaving tau, S and kept_cnt alone, when no threshold exists
// (NaN rows).
// (mt, st + lt): this thread's sweep-1 max and compensated sum.  ncand: the
// number of entries in A.cand when they include every kept entry, else -1.
template <typename TT, int NT>
__device__ __noinline__ bool adjust_row(const TT* row, int V, bool vec, float M, float c, int top_k,
                           float top_p, bool use_k, bool use_p, float mt, float st, float lt,
                           uint64_t pol, AdjShared& A, float& tau, float& S, uint32_t& kept_cnt,
                           int& ncand, unsigned long long* ctr) {
  // masses are pow2_neg(z) * 2^F with V * 2^F <= 2^62
  const int F = adj_mass_shift(V);
  const float fscale = adj_mass_scale(F);
  const double unscale = __longlong_as_double((long long)(1023 - F) << 52);
  uint32_t key = 0u, kc = kept_cnt;
  unsigned long long kept = 0ull;
  AdjGrid g{64.0f, 0.0f, true}, gw{64.0f, 0.0f, true};
  bool ok = false;
  ncand = -1;
  adj_count(ctr, kAdjRows);
  if constexpr (sizeof(TT) == 2) {
    if (use_k && top_k <= NT) {
      // The threads' sweep-1 maxima are top_k or more distinct entries at or
      // above the value where their count, from the top, reaches top_k: the
      // top-k edge (and a top-p edge, which lies inside the top-k set) is at or
      // above it.  The counting pass from there sees little more than the
      // top-k set and lists it for sweep 2.
      const uint32_t ktop = key16(M);
      for (int j = threadIdx.x; j < kAdjBins1; j += NT) A.cnt1[j] = 0u;
      __syncthreads();
      if (mt > -INFINITY) {
        const uint32_t j = ktop - key16(mt);  // mt <= M
        atomicAdd(&A.cnt1[j < (uint32_t)kAdjBins1 ? j : kAdjBins1 - 1], 1u);
      }
      __syncthreads();
      adj_select<NT>(A.cnt1, A.mass1, kAdjBins1, false, (uint32_t)top_k, 0.0, 0ull, A);
      const int sel = A.sel;
      __syncthreads();
      if (sel < kAdjBins1 - 1) {
        ok = adj_run_keys<NT, true>(reinterpret_cast<const __nv_bfloat16*>(row), V, vec, M, c, fscale,
                              top_k, top_p, use_k, use_p, 0ull, key16_value(ktop - sel), true,
                              pol, A, key, kept, kc, ncand);
        if (ok) adj_count(ctr, kAdjExact);
        else ncand = -1;
      }
    }
  }
  if (ok) {
    // resolved from the threads' maxima
  } else if (adj_estimate<TT, NT>(row, V, vec, M, c, S, top_k, top_p, use_k, use_p, pol, A, g, gw)) {
    if constexpr (sizeof(TT) == 2) {
      // bins of one value each, down to the window's cut (or the cut grid's)
      const float x_lo = M - (gw.lo > 0.0f ? gw.cut : g.cut) / c;
      if (key16(M) - key16(x_lo) < (uint32_t)kAdjBins1) {
        unsigned long long s_all = 0ull;
        bool fin = true;
        if (use_p && !use_k) {
          // the row's whole mass: every thread's compensated sum rescaled to
          // the row max, as an integer of the masses' scale (exact to add)
          const float f = ex2((mt - M) * c);
          const float a = st * f;
          const float r = lt * f + fmaf(st, f, -a);
          fin = !__syncthreads_or(!(a == a) || !(r == r));  // NaN logits: the general path
          const long long part = fin ? __float2ll_rn(a * fscale) + __float2ll_rn(r * fscale) : 0ll;
          s_all = adj_block_sum<NT>((unsigned long long)part, A);
        }
        if (fin) {
          int nc;
          ok = adj_run_keys<NT, false>(reinterpret_cast<const __nv_bfloat16*>(row), V, vec, M, c, fscale,
                                top_k, top_p, use_k, use_p, s_all, x_lo, false, pol, A, key, kept,
                                kc, nc);
          if (ok) adj_count(ctr, kAdjExact);
        }
      }
    }
    // the window grid first (when the sample gave one), then the cut grid
    if (!ok && gw.lo > 0.0f)
      ok = adj_run<TT, NT>(row, V, vec, M, c, fscale, top_k, top_p, use_k, use_p, gw, pol, A, key,
                           kept, kc, ctr);
    if (!ok)
      ok = adj_run<TT, NT>(row, V, vec, M, c, fscale, top_k, top_p, use_k, use_p, g, pol, A, key,
                           kept, kc, ctr);
    if (!ok) adj_count(ctr, kAdjMiss);
  } else {
    adj_count(ctr, kAdjTail);
  }
  if (!ok) {
    const AdjGrid full{64.0f, 0.0f, true};
    ok = adj_run<TT, NT>(row, V, vec, M, c, fscale, top_k, top_p, use_k, use_p, full, pol, A, key,
                         kept, kc, ctr);
  }
  if (!ok) {
    adj_count(ctr, kAdjNone);
    return false;
  }
  tau = key_value(key);
  S = (float)((double)kept * unscale);
  kept_cnt = kc;
  return true;
}

// kAdj: requests may carry top-k / top-p (P.topk, P.topp); their rows get a
// threshold tau and the kept mass as S before sweep 2.
template <typename TT, int NT, int MINB, bool kAdj = false>
__global__ void __launch_bounds__(NT, MINB) sweep_row_kernel(const Params P) {
  constexpr int NW = NT / 32;
  constexpr int kEl = 16 / sizeof(TT);
  __shared__ float4 red[2][NW];
  // adjusted rows: the selection's histograms, in dynamic shared memory
  // (sizeof(AdjShared) bytes at launch; none otherwise)
  extern __shared__ __align__(16) unsigned char adj_smem[];
  __shared__ long long s_slot;
  __shared__ int s_gmax, s_bad, s_prefix, s_x;
  __shared__ float s_dec[4];  // px, qx, flags
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, V = P.V;
  const bool vec = P.vec_ok != 0;

  if (tid == 0) {
    s_gmax = 0;
    s_bad = 0;
  }
  __syncthreads();
  {
    int gm = 0, bad = 0;
    for (int b = tid; b < B; b += NT) {
      const int g = __ldg(P.cu + b + 1) - __ldg(P.cu + b);
      gm = max(gm, g);
      bad |= (g < 0);
    }
    if (gm) atomicMax(&s_gmax, gm);
    if (bad) atomicOr(&s_bad, 1);
  }
  __syncthreads();
  if (blockIdx.x == 0 && tid == 0) {
    if (s_bad || __ldg(P.cu) != 0) set_err(P.err, SPECDEC_DEVERR_BAD_CU);
    *P.defer_count = 0;
  }
  const int64_t total = (int64_t)B * (s_gmax + 1);
  const uint64_t keep = policy_evict_last(), drop = policy_evict_first();

  for (int it = 0;; ++it) {
    // ---- thread 0 takes the next slot that has a row to verify -------------
    if (tid == 0) {
      long long u;
      int prefix = kPrefixAllAccepted;
      while (true) {
        u = (long long)atomicAdd(P.sched, 1ull);
        if (u >= total) break;
        const int i = (int)(u / B), b = (int)(u % B);
        const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
        if (i > g) continue;
        const int64_t t = (int64_t)c0 + b + i;
        if (t >= P.cap_rows) {
          set_err(P.err, SPECDEC_DEVERR_CAPACITY);
          continue;
        }
        prefix = i > 0 ? read_prefix(P.status, t - i, i, P.epoch) : kPrefixAllAccepted;
        if (i == g && prefix == kPrefixRejected) continue;  // bonus row nobody needs
        break;
      }
      s_slot = u;
      s_prefix = prefix;
    }
    __syncthreads();
    const long long u = s_slot;
    const int prefix = s_prefix;
    if (u >= total) break;
    const int i = (int)(u / B), b = (int)(u % B);
    const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
    const int64_t t = (int64_t)c0 + b + i, d = (int64_t)c0 + i;
    const bool has_q = i < g;
    // no draft rows: a one-hot drafter, q_i = [v == x_i] (never read)
    const bool onehot = P.q == nullptr;
    const TT* row = reinterpret_cast<const TT*>(P.logits) + t * (int64_t)V;
    const float* qrow = (has_q && !onehot) ? P.q + d * (int64_t)V : nullptr;
    const int par = it & 1;

    // thread 0 fetches what the accept test needs while sweep 1 runs
    int x = -1;
    float lx = 0.0f, qx = 0.0f;
    bool valid = true;
    if (tid == 0 && has_q) {
      x = __ldg(P.ids + d);
      valid = (x >= 0 && x < V);
      if (valid) {
        lx = load_logit(row + x);
        qx = onehot ? 1.0f : __ldg(qrow + x);
      }
      s_x = x;
    }

    // ---- sweep 1: (max, sum) ------------------------------------------------
    const int hi = vec ? V / kEl : V;
    float m0, s0, l0 = 0.0f;
    if constexpr (kAdj)
      sweep1_ff<TT, NT>(row, hi, vec, P.c, keep, m0, s0, l0);
    else
      sweep1<TT, NT>(row, 0, hi, vec, P.c, keep, m0, s0);
    const float mt = m0, st = s0;  // this thread's own (max, sum), for adjusted rows
    warp_softmax(m0, s0, P.c);
    if (lane == 0) red[par][warp] = make_float4(m0, s0, 0.f, 0.f);
    __syncthreads();
    float M = -INFINITY, S = 0.0f;
    for (int w = 0; w < NW; ++w) softmax_merge(M, S, red[par][w].x, red[par][w].y, P.c);
    float tau = -INFINITY;
    uint32_t kept_cnt = (uint32_t)V;
    int ncand = -1;  // adjusted rows: kept entries all in the candidate list
    if constexpr (kAdj) {
      const int kk = P.topk ? __ldg(P.topk + b) : 0;
      const float pp = P.topp ? __ldg(P.topp + b) : 1.0f;
      const bool use_k = kk >= 1 && kk < V, use_p = !(pp >= 1.0f);
      if ((use_k || use_p) && M > -INFINITY && M < INFINITY)
        adjust_row<TT, NT>(row, V, vec, M, P.c, kk, pp, use_k, use_p, mt, st, l0, keep,
                           *reinterpret_cast<AdjShared*>(adj_smem), tau, S, kept_cnt, ncand,
                           P.adj_ctr);
    }
    // few kept entries: at most 1/8 of the 16-byte vectors hold one, so sweep 2
    // skips the others (and their draft entries) instead of streaming them
    const bool sparse = kAdj && vec && (uint64_t)kept_cnt * (uint64_t)(8 * kEl) <= (uint64_t)V;
    const float invS = 1.0f / S;

    // ---- accept test (thread 0) and the race decision --------------------
    if (tid == 0) {
      float px = 0.0f;
      bool acc = false;
      if (has_q) {
        if (valid && lx >= tau) px = ex2((lx - M) * P.c) * invS;
        const float r = uniform_from_bits(uniform_bits(stream_key(P.seed, P.req_offset + b, i, 0), 0));
        acc = accept_test(r, px, qx);
      }
      // the earlier rows may have finished during sweep 1
      const int pfx = (prefix == kPrefixUnknown) ? read_prefix(P.status, t - i, i, P.epoch) : prefix;
      const bool race = (pfx == kPrefixAllAccepted) && (!has_q || !acc);
      s_dec[0] = px;
      s_dec[1] = qx;
      s_dec[2] = __int_as_float((acc ? 1 : 0) | (race ? 2 : 0) | (valid ? 0 : 4));
    }
    __syncthreads();
    const int flags = __float_as_int(s_dec[2]);
    const bool acc = flags & 1, race = flags & 2;
    const bool resid = has_q && !acc;
    const uint64_t rkey = stream_key(P.seed, P.req_offset + b, i, 1);

    // ---- sweep 2: beta and the race ---------------------------------------
    // (a one-hot draft needs no sweep for beta = p(x); only the race reads the
    // row again, with x removed from a correction's residual)
    float beta = 0.0f;
    Race best = race_none();
    if (kAdj && ncand >= 0) {
      const uint2* cand = reinterpret_cast<const AdjShared*>(adj_smem)->cand;
      if (has_q && !onehot && race)
        sweep2_list<NT, true, true>(cand, ncand, qrow, M, P.c, invS, tau, resid, rkey, beta, best, -1);
      else if (has_q && !onehot)
        sweep2_list<NT, true, false>(cand, ncand, qrow, M, P.c, invS, tau, resid, rkey, beta, best, -1);
      else if (race)
        sweep2_list<NT, false, true>(cand, ncand, qrow, M, P.c, invS, tau, resid, rkey, beta, best,
                                     resid ? s_x : -1);
    } else if (has_q && !onehot && race)
      sweep2<TT, NT, true, true, kAdj>(row, qrow, 0, hi, vec, M, P.c, invS, tau, resid, rkey, drop,
                                       beta, best, -1, sparse);
    else if (has_q && !onehot)
      sweep2<TT, NT, true, false, kAdj>(row, qrow, 0, hi, vec, M, P.c, invS, tau, resid, rkey, drop,
                                        beta, best, -1, sparse);
    else if (race)
      sweep2<TT, NT, false, true, kAdj>(row, qrow, 0, hi, vec, M, P.c, invS, tau, resid, rkey, drop,
                                        beta, best, resid ? s_x : -1, sparse);
    beta = warp_sum(beta);
    warp_race(best);
    if (lane == 0) red[par ^ 1][warp] = make_float4(beta, best.w, best.e, __int_as_float(best.idx));
    __syncthreads();
    if (tid == 0) {
      float bt = 0.0f;
      Race tb = race_none();
      for (int w = 0; w < NW; ++w) {
        const float4 r4 = red[par ^ 1][w];
        bt += r4.x;
        race_merge(tb, r4.y, r4.z, __float_as_int(r4.w));
      }
      P.row_stats[t] = make_float2(M, S);
      if (kAdj && P.row_tau) P.row_tau[t] = tau;
      uint32_t st = kStDone;
      if (has_q) {
        if (flags & 4) set_err(P.err, SPECDEC_DEVERR_BAD_DRAFT_ID);
        if (acc) st |= kStAccepted;
        if (P.out_beta) P.out_beta[d] = onehot ? s_dec[0] : bt;
        if (P.out_px) P.out_px[d] = s_dec[0];
        if (P.out_qx) P.out_qx[d] = s_dec[1];
        if (P.out_acc) P.out_acc[d] = acc ? 1 : 0;
      }
      if (race && tb.w > 0.0f) {
        P.out_tokens[t] = tb.idx;
        st |= kStRaceDone;
      }
      st_relaxed_u64(P.status + t, make_status(P.epoch, st));
    }
    // s_slot / s_dec / red[par] are rewritten next iteration only after the
    // __syncthreads that follows thread 0's next slot grab.
  }
}

// ---------------------------------------------------------------------------
// Dual row kernel (T > 0): every row is verified by two CTAs, neither of which
// ever waits for the other.  Each sweeps the whole target row once for (max,
// sum) (the second read of a row is served by L2, usually while the first is
// still in flight), so both hold bit-identical (M, S) and take the same accept
// test; each then runs sweep 2 over its half of the row.  Decisions that
// depend on timing (skipping a bonus row whose request already rejected,
// drawing the race) are taken once per row by whichever CTA gets there first
// (compare-and-swap on an epoch-tagged word); the halves' (beta, race) meet in
// global memory and the CTA that finishes second combines them, in a fixed
// order, and writes the row's outputs and status.  Work units are half rows
// handed out in position-major order, so half as many rows are live between
// their two sweeps as in the sweep kernel at the same CTA count.
// ---------------------------------------------------------------------------
constexpr uint32_t kDualSkip = 1u, kDualKeep = 2u, kDualRace = 1u, kDualNoRace = 2u;

// The row's decision for this call: the first caller's `want` (epoch-tagged).
__device__ __forceinline__ uint32_t dual_decide(unsigned long long* w, uint64_t epoch,
                                                uint32_t want) {
  const unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(w);
  if ((cur >> 8) == epoch) return (uint32_t)(cur & 0xFF);
  const unsigned long long mine = (epoch << 8) | want;
  const unsigned long long old = atomicCAS(w, cur, mine);
  return old == cur ? want : (uint32_t)(old & 0xFF);  // else the row's other CTA decided
}

template <typename TT>
__global__ void __launch_bounds__(512, 2) dual_row_kernel(const Params P) {
  constexpr int NT = 512, NW = NT / 32;
  constexpr int kEl = 16 / sizeof(TT);
  __shared__ float4 red[2][NW];
  __shared__ long long s_slot;
  __shared__ int s_gmax, s_bad, s_prefix;
  __shared__ float s_dec[4];  // px, qx, flags
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, V = P.V;
  const bool vec = P.vec_ok != 0;

  if (tid == 0) {
    s_gmax = 0;
    s_bad = 0;
  }
  __syncthreads();
  {
    int gm = 0, bad = 0;
    for (int b = tid; b < B; b += NT) {
      const int g = __ldg(P.cu + b + 1) - __ldg(P.cu + b);
      gm = max(gm, g);
      bad |= (g < 0);
    }
    if (gm) atomicMax(&s_gmax, gm);
    if (bad) atomicOr(&s_bad, 1);
  }
  __syncthreads();
  if (blockIdx.x == 0 && tid == 0) {
    if (s_bad || __ldg(P.cu) != 0) set_err(P.err, SPECDEC_DEVERR_BAD_CU);
    *P.defer_count = 0;
  }
  const int64_t total = 2 * (int64_t)B * (s_gmax + 1);  // half-row units
  const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
  const int nunits = vec ? V / kEl : V;
  const int halfu = (nunits + 1) / 2;

  for (int it = 0;; ++it) {
    // ---- thread 0 takes the next half row that has work ------------------
    if (tid == 0) {
      long long u;
      int prefix = kPrefixAllAccepted;
      while (true) {
        u = (long long)atomicAdd(P.sched, 1ull);
        if (u >= total) break;
        const long long r = u >> 1;
        const int i = (int)(r / B), b = (int)(r % B);
        const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
        if (i > g) continue;
        const int64_t t = (int64_t)c0 + b + i;
        if (t >= P.cap_rows) {
          set_err(P.err, SPECDEC_DEVERR_CAPACITY);
          continue;
        }
        prefix = i > 0 ? read_prefix(P.status, t - i, i, P.epoch) : kPrefixAllAccepted;
        if (i == g &&  // a bonus row nobody needs: both halves skip it or neither does
            dual_decide(P.dual_skip + t, P.epoch,
                        prefix == kPrefixRejected ? kDualSkip : kDualKeep) == kDualSkip)
          continue;
        break;
      }
      s_slot = u;
      s_prefix = prefix;
    }
    __syncthreads();
    const long long u = s_slot;
    const int prefix = s_prefix;
    if (u >= total) break;
    const int half = (int)(u & 1);
    const long long r = u >> 1;
    const int i = (int)(r / B), b = (int)(r % B);
    const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
    const int64_t t = (int64_t)c0 + b + i, d = (int64_t)c0 + i;
    const bool has_q = i < g;
    const TT* row = reinterpret_cast<const TT*>(P.logits) + t * (int64_t)V;
    const float* qrow = has_q ? P.q + d * (int64_t)V : nullptr;
    const int par = it & 1;

    int x = -1;
    float lx = 0.0f, qx = 0.0f;
    bool valid = true;
    if (tid == 0 && has_q) {
      x = __ldg(P.ids + d);
      valid = (x >= 0 && x < V);
      if (valid) {
        lx = load_logit(row + x);
        qx = __ldg(qrow + x);
      }
    }

    // ---- sweep 1 over the whole row --------------------------------------
    float m0, s0;
    sweep1<TT, NT>(row, 0, nunits, vec, P.c, keep, m0, s0);
    warp_softmax(m0, s0, P.c);
    if (lane == 0) red[par][warp] = make_float4(m0, s0, 0.f, 0.f);
    __syncthreads();
    float M = -INFINITY, S = 0.0f;
    for (int w = 0; w < NW; ++w) softmax_merge(M, S, red[par][w].x, red[par][w].y, P.c);
    const float invS = 1.0f / S;

    // ---- accept test (the same in both CTAs) and the row's race decision --
    if (tid == 0) {
      float px = 0.0f;
      bool acc = false;
      if (has_q) {
        if (valid) px = ex2((lx - M) * P.c) * invS;
        const float rr = uniform_from_bits(uniform_bits(stream_key(P.seed, P.req_offset + b, i, 0), 0));
        acc = accept_test(rr, px, qx);
      }
      const int pfx = (prefix == kPrefixUnknown) ? read_prefix(P.status, t - i, i, P.epoch) : prefix;
      const bool want = (pfx == kPrefixAllAccepted) && (!has_q || !acc);
      const bool race = dual_decide(P.dual_race + t, P.epoch, want ? kDualRace : kDualNoRace) ==
                        kDualRace;
      s_dec[0] = px;
      s_dec[1] = qx;
      s_dec[2] = __int_as_float((acc ? 1 : 0) | (race ? 2 : 0) | (valid ? 0 : 4));
    }
    __syncthreads();
    const int flags = __float_as_int(s_dec[2]);
    const bool acc = flags & 1, race = flags & 2;
    const bool resid = has_q && !acc;
    const uint64_t rkey = stream_key(P.seed, P.req_offset + b, i, 1);

    // ---- sweep 2 over this CTA's half ---------------------------------------
    const int lo = half ? halfu : 0, hi = half ? nunits : halfu;
    float beta = 0.0f;
    Race best = race_none();
    if (has_q && race)
      sweep2<TT, NT, true, true>(row, qrow, lo, hi, vec, M, P.c, invS, -INFINITY, resid, rkey, drop,
                                 beta, best);
    else if (has_q)
      sweep2<TT, NT, true, false>(row, qrow, lo, hi, vec, M, P.c, invS, -INFINITY, resid, rkey,
                                  drop, beta, best);
    else if (race)
      sweep2<TT, NT, false, true>(row, qrow, lo, hi, vec, M, P.c, invS, -INFINITY, resid, rkey,
                                  drop, beta, best);
    beta = warp_sum(beta);
    warp_race(best);
    if (lane == 0) red[par ^ 1][warp] = make_float4(beta, best.w, best.e, __int_as_float(best.idx));
    __syncthreads();
    if (tid == 0) {
      float bh = 0.0f;
      Race rh = race_none();
      for (int w = 0; w < NW; ++w) {
        const float4 r4 = red[par ^ 1][w];
        bh += r4.x;
        race_merge(rh, r4.y, r4.z, __float_as_int(r4.w));
      }
      P.dual_part[2 * t + half] = make_float4(bh, rh.w, rh.e, __int_as_float(rh.idx));
      __threadfence();
      if (atomicAdd(P.dual_cnt + t, 1) == 1) {  // second half done: combine
        __threadfence();
        const float4 h0 = __ldcg(P.dual_part + 2 * t), h1 = __ldcg(P.dual_part + 2 * t + 1);
        Race tb = race_none();
        race_merge(tb, h0.y, h0.z, __float_as_int(h0.w));
        race_merge(tb, h1.y, h1.z, __float_as_int(h1.w));
        P.row_stats[t] = make_float2(M, S);
        uint32_t st = kStDone;
        if (has_q) {
          if (flags & 4) set_err(P.err, SPECDEC_DEVERR_BAD_DRAFT_ID);
          if (acc) st |= kStAccepted;
          if (P.out_beta) P.out_beta[d] = h0.x + h1.x;
          if (P.out_px) P.out_px[d] = s_dec[0];
          if (P.out_qx) P.out_qx[d] = s_dec[1];
          if (P.out_acc) P.out_acc[d] = acc ? 1 : 0;
        }
        if (race && tb.w > 0.0f) {
          P.out_tokens[t] = tb.idx;
          st |= kStRaceDone;
        }
        P.dual_cnt[t] = 0;  // ready for the next call
        st_relaxed_u64(P.status + t, make_status(P.epoch, st));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Pair row kernel (T > 0): the sweep kernel with every row split over a cluster
// of two CTAs (512 threads each, two CTAs per SM).  Rank 0 takes the work slot
// and sends it to both CTAs; each CTA sweeps half of the row; the halves'
// (max, sum) and rank 0's view of the request's earlier rows are exchanged
// through distributed shared memory, so both CTAs take the same accept / race
// decision; the halves' beta and race candidates go to rank 0, which writes the
// outputs.  Half as many rows are live in L2 between their two sweeps as with
// one row per CTA at the same number of threads per SM.
// ---------------------------------------------------------------------------
struct alignas(16) PairShared {
  uint64_t bdesc[2];   // work slot arrived (1 arrival, from rank 0)
  uint64_t bms[2];     // both halves' (max, sum) arrived (2 arrivals)
  uint64_t bred[2];    // both halves' (beta, race) arrived at rank 0 (2 arrivals)
  float4 desc[2];      // (slot lo bits, slot hi bits, prefix at grab, -)
  float4 ms[2][2];     // [parity][rank] (max, sum, rank 0's prefix, -)
  float4 part[2][2];   // [parity][rank] (beta, race w, race e, race index)
  float4 red[2][16];
  float dec[4];        // max, sum, flags, -
  float acc_x[2];      // p(x), q(x)
  int gmax, bad, flag;
};

template <typename TT, int NT = 512>
__global__ void __launch_bounds__(NT, 1024 / NT) pair_row_kernel(const Params P) {
  constexpr int NW = NT / 32;
  static_assert(NW <= 16, "PairShared::red holds 16 warps");
  constexpr int kEl = 16 / sizeof(TT);
  __shared__ PairShared S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const uint32_t cid = cluster_id_x();
  const int B = P.B, V = P.V;
  const bool vec = P.vec_ok != 0;

  if (tid == 0) {
    for (int p = 0; p < 2; ++p) {
      mbar_init(smem_addr(&S.bdesc[p]), 1);
      mbar_init(smem_addr(&S.bms[p]), 2);
      mbar_init(smem_addr(&S.bred[p]), 2);
    }
    S.gmax = 0;
    S.bad = 0;
    S.flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  {
    int gm = 0, bad = 0;
    for (int b = tid; b < B; b += NT) {
      const int g = __ldg(P.cu + b + 1) - __ldg(P.cu + b);
      gm = max(gm, g);
      bad |= (g < 0);
    }
    if (gm) atomicMax(&S.gmax, gm);
    if (bad) atomicOr(&S.bad, 1);
  }
  cluster_sync_all();
  if (cid == 0 && rank == 0 && tid == 0) {
    if (S.bad || __ldg(P.cu) != 0) set_err(P.err, SPECDEC_DEVERR_BAD_CU);
    *P.defer_count = 0;
  }
  const int64_t total = (int64_t)B * (S.gmax + 1);
  const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
  const int nunits = vec ? V / kEl : V;
  const int half = (nunits + 1) / 2;
  const int lo = rank ? half : 0, hi = rank ? nunits : half;
  const uint64_t limit = P.wait_ns ? P.wait_ns : kWaitLimitNs;
  bool ok = true;

  // ---- rank 0 takes a slot and sends it to both CTAs' desc[p] -------------
  // Row k + 1's slot is taken by thread 32 of rank 0 right after row k's final
  // block barrier, while thread 0 still combines the halves and writes row k's
  // outputs, so the two latencies overlap.
  auto grab = [&](int p, bool first) {
    long long u;
    int prefix = kPrefixAllAccepted;
    while (true) {
      u = (long long)atomicAdd(P.sched, 1ull);
      if (u >= total) {
        u = -1;
        break;
      }
      const int i = (int)(u / B), b = (int)(u % B);
      const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
      if (i > g) continue;
      const int64_t t = (int64_t)c0 + b + i;
      if (t >= P.cap_rows) {
        set_err(P.err, SPECDEC_DEVERR_CAPACITY);
        continue;
      }
      prefix = i > 0 ? read_prefix(P.status, t - i, i, P.epoch) : kPrefixAllAccepted;
      if (i == g && prefix == kPrefixRejected) continue;  // bonus row nobody needs
      break;
    }
    const uint32_t slot = smem_addr(&S.desc[p]);
    for (uint32_t r = 0; r < 2; ++r) {
      if (P.stall_peer && r == 1 && first) continue;  // test hook: rank 1 is left waiting
      st_cluster_v4(mapa(slot, r), __int_as_float((int)(u & 0xFFFFFFFF)),
                    __int_as_float((int)(u >> 32)), __int_as_float(prefix), 0.f);
      mbar_arrive_cluster(mapa(smem_addr(&S.bdesc[p]), r));
    }
  };
  if (rank == 0 && tid == 0) grab(0, true);

  for (uint32_t k = 0;; ++k) {
    const int par = k & 1;
    const uint32_t ph = (k >> 1) & 1;
    if (tid == 0) S.flag = (ok && mbar_wait_cluster(smem_addr(&S.bdesc[par]), ph, limit)) ? 0 : 1;
    __syncthreads();
    if (S.flag) {
      ok = false;
      break;
    }
    const float4 dsc = S.desc[par];
    const long long u = (long long)(((unsigned long long)(uint32_t)__float_as_int(dsc.y) << 32) |
                                    (uint32_t)__float_as_int(dsc.x));
    if (u < 0) break;
    const int prefix0 = __float_as_int(dsc.z);
    const int i = (int)(u / B), b = (int)(u % B);
    const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
    const int64_t t = (int64_t)c0 + b + i, d = (int64_t)c0 + i;
    const bool has_q = i < g;
    const TT* row = reinterpret_cast<const TT*>(P.logits) + t * (int64_t)V;
    const float* qrow = has_q ? P.q + d * (int64_t)V : nullptr;

    int x = -1;
    float lx = 0.0f, qx = 0.0f;
    bool valid = true;
    if (tid == 0 && has_q) {
      x = __ldg(P.ids + d);
      valid = (x >= 0 && x < V);
      if (valid) {
        lx = load_logit(row + x);
        qx = __ldg(qrow + x);
      }
    }

    // ---- sweep 1 over this CTA's half -----------------------------------------
    float m0, s0;
    sweep1<TT, NT>(row, lo, hi, vec, P.c, keep, m0, s0);
    warp_softmax(m0, s0, P.c);
    if (lane == 0) S.red[0][warp] = make_float4(m0, s0, 0.f, 0.f);
    __syncthreads();
    if (tid == 0) {
      float mh = -INFINITY, sh = 0.0f;
      for (int w = 0; w < NW; ++w) softmax_merge(mh, sh, S.red[0][w].x, S.red[0][w].y, P.c);
      int pfx = prefix0;
      if (rank == 0 && pfx == kPrefixUnknown) pfx = read_prefix(P.status, t - i, i, P.epoch);
      const uint32_t slot = smem_addr(&S.ms[par][rank]);
      for (uint32_t r = 0; r < 2; ++r) {
        st_cluster_v4(mapa(slot, r), mh, sh, __int_as_float(pfx), 0.f);
        mbar_arrive_cluster(mapa(smem_addr(&S.bms[par]), r));
      }
      ok = mbar_wait_cluster(smem_addr(&S.bms[par]), ph, limit);
      float M = -INFINITY, Ssum = 0.0f;
      softmax_merge(M, Ssum, S.ms[par][0].x, S.ms[par][0].y, P.c);
      softmax_merge(M, Ssum, S.ms[par][1].x, S.ms[par][1].y, P.c);
      const int prefix = __float_as_int(S.ms[par][0].z);
      const float invS = 1.0f / Ssum;
      float px = 0.0f;
      bool acc = false;
      if (has_q) {
        if (valid) px = ex2((lx - M) * P.c) * invS;
        const float r = uniform_from_bits(uniform_bits(stream_key(P.seed, P.req_offset + b, i, 0), 0));
        acc = accept_test(r, px, qx);
      }
      const bool race = (prefix == kPrefixAllAccepted) && (!has_q || !acc);
      S.dec[0] = M;
      S.dec[1] = Ssum;
      S.dec[2] = __int_as_float((acc ? 1 : 0) | (race ? 2 : 0) | (valid ? 0 : 4) | (ok ? 0 : 8));
      S.acc_x[0] = px;
      S.acc_x[1] = qx;
    }
    __syncthreads();
    const float M = S.dec[0], Ssum = S.dec[1];
    const int flags = __float_as_int(S.dec[2]);
    if (flags & 8) {
      ok = false;
      break;
    }
    const float invS = 1.0f / Ssum;
    const bool acc = flags & 1, race = flags & 2;
    const bool resid = has_q && !acc;
    const uint64_t rkey = stream_key(P.seed, P.req_offset + b, i, 1);

    // ---- sweep 2 over this CTA's half -----------------------------------------
    float beta = 0.0f;
    Race best = race_none();
    if (has_q && race)
      sweep2<TT, NT, true, true>(row, qrow, lo, hi, vec, M, P.c, invS, -INFINITY, resid, rkey, drop,
                                 beta, best);
    else if (has_q)
      sweep2<TT, NT, true, false>(row, qrow, lo, hi, vec, M, P.c, invS, -INFINITY, resid, rkey, drop,
                                  beta, best);
    else if (race)
      sweep2<TT, NT, false, true>(row, qrow, lo, hi, vec, M, P.c, invS, -INFINITY, resid, rkey, drop,
                                  beta, best);
    beta = warp_sum(beta);
    warp_race(best);
    if (lane == 0) S.red[1][warp] = make_float4(beta, best.w, best.e, __int_as_float(best.idx));
    __syncthreads();
    // both CTAs have read desc[par ^ 1] (row k - 1) before this row's first barrier
    if (rank == 0 && tid == 32) grab(par ^ 1, false);
    if (tid == 0) {
      float bh = 0.0f;
      Race rh = race_none();
      for (int w = 0; w < NW; ++w) {
        const float4 r4 = S.red[1][w];
        bh += r4.x;
        race_merge(rh, r4.y, r4.z, __float_as_int(r4.w));
      }
      st_cluster_v4(mapa(smem_addr(&S.part[par][rank]), 0), bh, rh.w, rh.e, __int_as_float(rh.idx));
      mbar_arrive_cluster(mapa(smem_addr(&S.bred[par]), 0));
      if (rank == 0) {
        ok = mbar_wait_cluster(smem_addr(&S.bred[par]), ph, limit);
        float bt = 0.0f;
        Race tb = race_none();
        for (int r = 0; r < 2; ++r) {
          const float4 r4 = S.part[par][r];
          bt += r4.x;
          race_merge(tb, r4.y, r4.z, __float_as_int(r4.w));
        }
        if (ok) {
          P.row_stats[t] = make_float2(M, Ssum);
          uint32_t stw = kStDone;
          if (has_q) {
            if (flags & 4) set_err(P.err, SPECDEC_DEVERR_BAD_DRAFT_ID);
            if (acc) stw |= kStAccepted;
            if (P.out_beta) P.out_beta[d] = bt;
            if (P.out_px) P.out_px[d] = S.acc_x[0];
            if (P.out_qx) P.out_qx[d] = S.acc_x[1];
            if (P.out_acc) P.out_acc[d] = acc ? 1 : 0;
          }
          if (race && tb.w > 0.0f) {
            P.out_tokens[t] = tb.idx;
            stw |= kStRaceDone;
          }
          st_relaxed_u64(P.status + t, make_status(P.epoch, stw));
        }
      }
    }
  }
  if (!ok && tid == 0) set_err(P.err, SPECDEC_DEVERR_TIMEOUT);
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its peer may still write to its shared memory
}

// ---------------------------------------------------------------------------
// Streamed row kernel (T > 0): the sweep kernel's two sweeps, fed by bulk copies
// through a shared-memory ring instead of register-held loads.  One CTA per SM:
// a producer thread takes work slots (position-major, global counter), publishes
// a row descriptor and issues, in a fixed order, the 16 KB stages of sweep 1
// (target row, L2 evict_last) and of sweep 2 (target row again from L2 plus the
// draft row, evict_first); it runs ahead across rows as far as the ring allows.
// Sixteen consumer warps follow the same order.  Their reductions and decisions
// between sweeps do not stop the copies, so HBM keeps streaming.
// ---------------------------------------------------------------------------
constexpr int kStreamConsumerWarps = 16;
constexpr int kStreamConsumers = kStreamConsumerWarps * 32;
constexpr int kStreamThreads = kStreamConsumers + 32;
constexpr int kStageBytes = 16384;
constexpr int kMaxStages = 16;
constexpr int kDescSlots = 4;

struct alignas(16) StreamShared {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t dfull[kDescSlots];
  uint64_t dempty[kDescSlots];
  long long desc_u[kDescSlots];     // work slot, or -1 = no more work
  int desc_prefix[kDescSlots];      // prefix state read when the slot was taken
  float4 red[2][kStreamConsumerWarps];
  float dec[4];
  int gmax, bad;
  volatile int abort_flag;
};

__device__ __forceinline__ bool stream_wait(StreamShared& S, uint32_t bar, uint32_t parity) {
  if (S.abort_flag) return false;
  if (mbar_wait(bar, parity)) return true;
  S.abort_flag = 1;
  return false;
}

template <typename TT, int MINB>
__global__ void __launch_bounds__(kStreamThreads, MINB) stream_row_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  constexpr int kEl1 = kStageBytes / sizeof(TT);  // target elements per stage
  constexpr int kQPerGroup = kEl1 / 4096;         // draft stages per sweep-2 group (2 bf16, 1 f32)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, V = P.V;
  const int NS = P.nq;
  unsigned char* ring = smem_raw;
  StreamShared& S = *reinterpret_cast<StreamShared*>(smem_raw + (size_t)NS * kStageBytes);
  const int n1 = (V + kEl1 - 1) / kEl1;                   // target stages per sweep
  const int nq = (V + 4095) / 4096;                       // draft stages per row

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&S.full[s]), 1);
      mbar_init(smem_addr(&S.empty[s]), kStreamConsumerWarps);
    }
    for (int s = 0; s < kDescSlots; ++s) {
      mbar_init(smem_addr(&S.dfull[s]), 1);
      mbar_init(smem_addr(&S.dempty[s]), 1);
    }
    S.gmax = 0;
    S.bad = 0;
    S.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  {
    int gm = 0, bad = 0;
    for (int b = tid; b < B; b += blockDim.x) {
      const int g = __ldg(P.cu + b + 1) - __ldg(P.cu + b);
      gm = max(gm, g);
      bad |= (g < 0);
    }
    if (gm) atomicMax(&S.gmax, gm);
    if (bad) atomicOr(&S.bad, 1);
  }
  __syncthreads();
  if (blockIdx.x == 0 && tid == 0) {
    if (S.bad || __ldg(P.cu) != 0) set_err(P.err, SPECDEC_DEVERR_BAD_CU);
    *P.defer_count = 0;
  }
  const int64_t total = (int64_t)B * (S.gmax + 1);

  if (warp == kStreamConsumerWarps) {
    // ===================== producer ==========================================
    if (lane == 0) {
      const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
      uint32_t fill = 0, k = 0;
      auto issue = [&](const void* src, int bytes, uint64_t pol) -> bool {
        const int s = fill % NS;
        if (!stream_wait(S, smem_addr(&S.empty[s]), ((fill / NS) & 1) ^ 1)) return false;
        mbar_arrive_expect_tx(smem_addr(&S.full[s]), bytes);
        bulk_load(smem_addr(ring + (size_t)s * kStageBytes), src, bytes, smem_addr(&S.full[s]), pol);
        ++fill;
        return true;
      };
      for (;; ++k) {
        long long u;
        int prefix = kPrefixAllAccepted;
        while (true) {
          u = (long long)atomicAdd(P.sched, 1ull);
          if (u >= total) {
            u = -1;
            break;
          }
          const int i = (int)(u / B), b = (int)(u % B);
          const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
          if (i > g) continue;
          const int64_t t = (int64_t)c0 + b + i;
          if (t >= P.cap_rows) {
            set_err(P.err, SPECDEC_DEVERR_CAPACITY);
            continue;
          }
          prefix = i > 0 ? read_prefix(P.status, t - i, i, P.epoch) : kPrefixAllAccepted;
          if (i == g && prefix == kPrefixUnknown) {
            // A bonus row is needed only when every draft was accepted: give the
            // rows still in flight (on other SMs, never blocked) a bounded time.
            const uint64_t t0 = globaltimer_ns();
            while (prefix == kPrefixUnknown && globaltimer_ns() - t0 < 200000ull) {
              __nanosleep(500);
              prefix = read_prefix(P.status, t - i, i, P.epoch);
            }
          }
          if (i == g && prefix == kPrefixRejected) continue;  // bonus row nobody needs
          break;
        }
        const int ds = k % kDescSlots;
        if (!stream_wait(S, smem_addr(&S.dempty[ds]), ((k / kDescSlots) & 1) ^ 1)) u = -1;
        S.desc_u[ds] = S.abort_flag ? -1 : u;
        S.desc_prefix[ds] = prefix;
        mbar_arrive(smem_addr(&S.dfull[ds]));
        if (u < 0 || S.abort_flag) break;
        const int i = (int)(u / B), b = (int)(u % B);
        const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
        const int64_t t = (int64_t)c0 + b + i, d = (int64_t)c0 + i;
        const bool has_q = i < g;
        const TT* row = reinterpret_cast<const TT*>(P.logits) + t * (int64_t)V;
        const float* qrow = P.q + d * (int64_t)V;
        bool ok = true;
        for (int c = 0; c < n1 && ok; ++c)
          ok = issue(row + (size_t)c * kEl1, min(kEl1, V - c * kEl1) * (int)sizeof(TT), keep);
        for (int c = 0; c < n1 && ok; ++c) {
          ok = issue(row + (size_t)c * kEl1, min(kEl1, V - c * kEl1) * (int)sizeof(TT), drop);
          if (has_q)
            for (int h = 0; h < kQPerGroup && ok; ++h) {
              const int qc = c * kQPerGroup + h;
              if (qc < nq) ok = issue(qrow + (size_t)qc * 4096, min(4096, V - qc * 4096) * 4, drop);
            }
        }
        if (!ok) break;
      }
      if (S.abort_flag) {
        set_err(P.err, SPECDEC_DEVERR_TIMEOUT);
        // let every issued copy land before the CTA may exit
        for (uint32_t f = fill > (uint32_t)NS ? fill - NS : 0; f < fill; ++f)
          mbar_wait(smem_addr(&S.full[f % NS]), (f / NS) & 1);
        for (int s = 0; s < kDescSlots; ++s) {  // release consumers waiting for a row
          S.desc_u[s] = -1;
          mbar_arrive(smem_addr(&S.dfull[s]));
        }
      }
    }
    __syncwarp();
    return;
  }

  // ===================== consumers ===========================================
  uint32_t cc = 0;
  for (uint32_t k = 0;; ++k) {
    const int ds = k % kDescSlots;
    bool ok = stream_wait(S, smem_addr(&S.dfull[ds]), (k / kDescSlots) & 1);
    const long long u = ok ? S.desc_u[ds] : -1;
    const int prefix0 = S.desc_prefix[ds];
    if (named_bar_or(1, kStreamConsumers, u < 0)) break;
    const int i = (int)(u / B), b = (int)(u % B);
    const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
    const int64_t t = (int64_t)c0 + b + i, d = (int64_t)c0 + i;
    const bool has_q = i < g;
    const int par = k & 1;

    int x = -1;
    float lx = 0.0f, qx = 0.0f;
    bool valid = true;
    if (tid == 0 && has_q) {
      x = __ldg(P.ids + d);
      valid = (x >= 0 && x < V);
      if (valid) {
        lx = load_logit(reinterpret_cast<const TT*>(P.logits) + t * (int64_t)V + x);
        qx = __ldg(P.q + d * (int64_t)V + x);
      }
    }

    // ---- sweep 1 ------------------------------------------------------------
    float m0 = -INFINITY, s0 = 0.0f;
    for (int c = 0; c < n1; ++c, ++cc) {
      const int s = cc % NS;
      ok &= stream_wait(S, smem_addr(&S.full[s]), (cc / NS) & 1);
      const int nvec = min(kEl1, V - c * kEl1) * (int)sizeof(TT) / 16;
      const uint4* st = reinterpret_cast<const uint4*>(ring + (size_t)s * kStageBytes);
      for (int j = tid; j < nvec; j += kStreamConsumers) softmax_acc16<TT>(st[j], m0, s0, P.c);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.empty[s]));
    }
    warp_softmax(m0, s0, P.c);
    if (lane == 0) S.red[par][warp] = make_float4(m0, s0, 0.f, 0.f);
    named_bar_sync(1, kStreamConsumers);
    float M = -INFINITY, Ssum = 0.0f;
    for (int w = 0; w < kStreamConsumerWarps; ++w) softmax_merge(M, Ssum, S.red[par][w].x, S.red[par][w].y, P.c);
    const float invS = 1.0f / Ssum;

    if (tid == 0) {
      const int prefix = (i > 0 && prefix0 == kPrefixUnknown)
                             ? read_prefix(P.status, t - i, i, P.epoch) : prefix0;
      float px = 0.0f;
      bool acc = false;
      if (has_q) {
        if (valid) px = ex2((lx - M) * P.c) * invS;
        const float r = uniform_from_bits(uniform_bits(stream_key(P.seed, P.req_offset + b, i, 0), 0));
        acc = accept_test(r, px, qx);
      }
      const bool race = (prefix == kPrefixAllAccepted) && (!has_q || !acc);
      S.dec[0] = px;
      S.dec[1] = qx;
      S.dec[2] = __int_as_float((acc ? 1 : 0) | (race ? 2 : 0) | (valid ? 0 : 4));
    }
    named_bar_sync(1, kStreamConsumers);
    const int flags = __float_as_int(S.dec[2]);
    const bool acc = flags & 1, race = flags & 2;
    const bool resid = has_q && !acc;
    const uint64_t rkey = stream_key(P.seed, P.req_offset + b, i, 1);

    // ---- sweep 2: groups of one target stage and its draft stages ------------
    float beta = 0.0f;
    Race best = race_none();
    for (int c = 0; c < n1; ++c) {
      const int ne = min(kEl1, V - c * kEl1);
      const int st_t = cc % NS;
      ok &= stream_wait(S, smem_addr(&S.full[st_t]), (cc / NS) & 1);
      ++cc;
      int st_q[kQPerGroup];
      int nqs = 0;
      if (has_q) {
        for (int h = 0; h < kQPerGroup; ++h)
          if (c * kQPerGroup + h < nq) {
            st_q[h] = cc % NS;
            ok &= stream_wait(S, smem_addr(&S.full[st_q[h]]), (cc / NS) & 1);
            ++cc;
            ++nqs;
          }
      }
      if (has_q || race) {
        const unsigned char* tst = ring + (size_t)st_t * kStageBytes;
        for (int e4 = tid; e4 * 4 < ne; e4 += kStreamConsumers) {
          float l[4];
          if constexpr (sizeof(TT) == 2) {
            const uint2 w = reinterpret_cast<const uint2*>(tst)[e4];
            l[0] = bf16_lo(w.x); l[1] = bf16_hi(w.x); l[2] = bf16_lo(w.y); l[3] = bf16_hi(w.y);
          } else {
            const float4 w = reinterpret_cast<const float4*>(tst)[e4];
            l[0] = w.x; l[1] = w.y; l[2] = w.z; l[3] = w.w;
          }
          float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
          if (has_q)
            q4 = reinterpret_cast<const float4*>(ring + (size_t)st_q[e4 >> 10] * kStageBytes)[e4 & 1023];
          const uint32_t v = (uint32_t)(c * kEl1 + 4 * e4);
          if (has_q && race)
            sweep2_4<true, true, false>(l, q4, M, P.c, invS, -INFINITY, resid, rkey, v, beta, best);
          else if (has_q)
            sweep2_4<true, false, false>(l, q4, M, P.c, invS, -INFINITY, resid, rkey, v, beta, best);
          else
            sweep2_4<false, true, false>(l, q4, M, P.c, invS, -INFINITY, resid, rkey, v, beta, best);
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&S.empty[st_t]));
        for (int h = 0; h < nqs; ++h) mbar_arrive(smem_addr(&S.empty[st_q[h]]));
      }
    }
    beta = warp_sum(beta);
    warp_race(best);
    if (lane == 0) S.red[par ^ 1][warp] = make_float4(beta, best.w, best.e, __int_as_float(best.idx));
    named_bar_sync(1, kStreamConsumers);
    if (tid == 0) {
      float bt = 0.0f;
      Race tb = race_none();
      for (int w = 0; w < kStreamConsumerWarps; ++w) {
        const float4 r4 = S.red[par ^ 1][w];
        bt += r4.x;
        race_merge(tb, r4.y, r4.z, __float_as_int(r4.w));
      }
      if (ok) {
        P.row_stats[t] = make_float2(M, Ssum);
        uint32_t stw = kStDone;
        if (has_q) {
          if (flags & 4) set_err(P.err, SPECDEC_DEVERR_BAD_DRAFT_ID);
          if (acc) stw |= kStAccepted;
          if (P.out_beta) P.out_beta[d] = bt;
          if (P.out_px) P.out_px[d] = S.dec[0];
          if (P.out_qx) P.out_qx[d] = S.dec[1];
          if (P.out_acc) P.out_acc[d] = acc ? 1 : 0;
        }
        if (race && tb.w > 0.0f) {
          P.out_tokens[t] = tb.idx;
          stw |= kStRaceDone;
        }
        st_relaxed_u64(P.status + t, make_status(P.epoch, stw));
      }
      mbar_arrive(smem_addr(&S.dempty[ds]));
    }
    if (named_bar_or(1, kStreamConsumers, !ok)) {
      if (tid == 0) set_err(P.err, SPECDEC_DEVERR_TIMEOUT);
      break;
    }
  }
}

// ---------------------------------------------------------------------------
// Two-pass path (T > 0): statistics of every target row, then one block per
// draft row for beta and the accept test.  Grid-stride loops, so the grid does
// not depend on N_t (read from cu[B] on the device).
// ---------------------------------------------------------------------------
constexpr int kRowThreads = 256;

template <typename T>
__device__ __forceinline__ void block_softmax(float& m, float& s, float c, float4* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  warp_softmax(m, s, c);
  __syncthreads();
  if (lane == 0) red[warp] = make_float4(m, s, 0.f, 0.f);
  __syncthreads();
  m = -INFINITY;
  s = 0.0f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) softmax_merge(m, s, red[w].x, red[w].y, c);
}

template <typename TT>
__global__ void __launch_bounds__(kRowThreads) stats_kernel(const Params P) {
  __shared__ float4 red[kRowThreads / 32];
  const int B = P.B, V = P.V;
  const int64_t n_t = (int64_t)__ldg(P.cu + B) + B;
  const int64_t rows = min(n_t, P.cap_rows);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (n_t > P.cap_rows) set_err(P.err, SPECDEC_DEVERR_CAPACITY);
    if (P.defer_count) *P.defer_count = 0;
  }
  for (int64_t t = blockIdx.x; t < rows; t += gridDim.x) {
    const TT* row = reinterpret_cast<const TT*>(P.logits) + t * (int64_t)V;
    float m = -INFINITY, s = 0.0f;
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
      const float x = load_logit(row + v);
      if (x > m) {
        s *= ex2((m - x) * P.c);
        m = x;
      }
      if (m != -INFINITY) s += ex2((x - m) * P.c);
    }
    block_softmax<TT>(m, s, P.c, red);
    if (threadIdx.x == 0) P.row_stats[t] = make_float2(m, s);
    __syncthreads();
  }
}

template <typename TT>
__global__ void __launch_bounds__(kRowThreads) verify_kernel(const Params P) {
  __shared__ float red[kRowThreads / 32];
  const int B = P.B, V = P.V;
  const int64_t n_d = __ldg(P.cu + B);
  for (int64_t d = blockIdx.x; d < n_d; d += gridDim.x) {
    const int b = request_of_draft(P.cu, B, d);
    const int c0 = __ldg(P.cu + b);
    const int i = (int)(d - c0);
    const int64_t t = d + b;
    if (t >= P.cap_rows || i < 0) continue;
    const float2 ms = P.row_stats[t];
    const float invS = 1.0f / ms.y;
    const TT* row = reinterpret_cast<const TT*>(P.logits) + t * (int64_t)V;
    const float* qrow = P.q + d * (int64_t)V;
    float beta = 0.0f;
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
      const float p = ex2((load_logit(row + v) - ms.x) * P.c) * invS;
      beta += fminf(p, __ldg(qrow + v));
    }
    beta = warp_sum(beta);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = beta;
    __syncthreads();
    if (threadIdx.x == 0) {
      float bt = 0.0f;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) bt += red[w];
      const int x = __ldg(P.ids + d);
      const bool valid = (x >= 0 && x < V);
      float px = 0.0f, qx = 0.0f;
      if (valid) {
        px = ex2((load_logit(row + x) - ms.x) * P.c) * invS;
        qx = __ldg(qrow + x);
      } else {
        set_err(P.err, SPECDEC_DEVERR_BAD_DRAFT_ID);
      }
      const float r = uniform_from_bits(uniform_bits(stream_key(P.seed, P.req_offset + b, i, 0), 0));
      const bool acc = accept_test(r, px, qx);
      if (P.out_beta) P.out_beta[d] = bt;
      if (P.out_px) P.out_px[d] = px;
      if (P.out_qx) P.out_qx[d] = qx;
      if (P.out_acc) P.out_acc[d] = acc ? 1 : 0;
      st_relaxed_u64(P.status + t, make_status(P.epoch, kStDone | (acc ? kStAccepted : 0u)));
    }
  }
}

// ---------------------------------------------------------------------------
// First-rejection scan per request (T > 0): n_b, accepted drafts, -1 tail, and
// the list of requests whose extra token the race kernel still has to draw.
// ---------------------------------------------------------------------------
static __global__ void finalize_kernel(const Params P) {
  wait_for_previous_kernel();
  const int B = P.B;
  if (blockIdx.x == 0 && threadIdx.x == 0 && P.sched) *P.sched = 0ull;
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
    const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
    const int64_t t0 = (int64_t)c0 + b;
    if (g < 0 || t0 + g >= P.cap_rows) continue;
    int n = g;
    for (int i = 0; i < g; ++i) {
      const uint64_t st = P.status[t0 + i];
      if ((st >> 8) != P.epoch || !(st & kStDone)) {  // row never verified (aborted launch)
        set_err(P.err, SPECDEC_DEVERR_TIMEOUT);
        n = i;
        break;
      }
      if (!(st & kStAccepted)) {
        n = i;
        break;
      }
    }
    P.out_nacc[b] = n;
    for (int i = 0; i < n; ++i) P.out_tokens[t0 + i] = __ldg(P.ids + c0 + i);
    for (int i = n + 1; i <= g; ++i) P.out_tokens[t0 + i] = -1;
    const uint64_t st = P.status[t0 + n];
    if (!((st >> 8) == P.epoch && (st & kStRaceDone))) {
      P.ws_nacc[b] = n;
      const int k = atomicAdd(P.defer_count, 1);
      P.defer_list[k] = b;
    }
  }
}

// ---------------------------------------------------------------------------
// Race for deferred requests: re-reads row (b, n_b) (and the draft row when it
// is a correction), split into slices over several CTAs.  Each CTA writes the
// best candidate of its slice; the last CTA of a request (counted with an
// atomic) merges them and writes the token.  When the residual max(0, p - q) is
// zero everywhere (reachable only through rounding) that CTA races over p.
// ---------------------------------------------------------------------------
template <typename TT>
__device__ __forceinline__ Race block_race(Race best, float4* red) {
  warp_race(best);
  __syncthreads();
  if ((threadIdx.x & 31) == 0)
    red[threadIdx.x >> 5] = make_float4(best.w, best.e, __int_as_float(best.idx), 0.f);
  __syncthreads();
  Race tb = race_none();
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) race_merge(tb, red[w].x, red[w].y, __float_as_int(red[w].z));
  return tb;
}

template <typename TT>
__global__ void __launch_bounds__(kRowThreads) race_kernel(const Params P) {
  __shared__ float4 red[kRowThreads / 32];
  __shared__ int s_last;
  wait_for_previous_kernel();
  const int V = P.V;
  const int count = *P.defer_count;
  const int S = P.rslices;
  for (int64_t item = blockIdx.x; item < (int64_t)count * S; item += gridDim.x) {
    const int k = (int)(item / S), sl = (int)(item % S);
    const int b = P.defer_list[k];
    const int n = P.ws_nacc[b];
    const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
    const int64_t t = (int64_t)c0 + b + n;
    const bool has_q = n < g;
    const float2 ms = P.row_stats[t];
    const float invS = 1.0f / ms.y;
    const float tau = P.row_tau ? P.row_tau[t] : -INFINITY;  // adjusted rows keep l >= tau
    const TT* row = reinterpret_cast<const TT*>(P.logits) + t * (int64_t)V;
    const bool onehot = P.q == nullptr;
    const float* qrow = (has_q && !onehot) ? P.q + ((int64_t)c0 + n) * (int64_t)V : nullptr;
    const int excl = (has_q && onehot) ? __ldg(P.ids + c0 + n) : -1;  // residual of a one-hot draft
    const uint64_t rkey = stream_key(P.seed, P.req_offset + b, n, 1);
    const int v0 = sl * P.rslice_len, v1 = min(V, v0 + P.rslice_len);
    // Visits the slice's (weight, index) pairs: 16-byte loads where rows are
    // 16-byte aligned (v0 is a multiple of 8), elements otherwise.
    auto weight = [&](float xv, float qv, int v) {
      const float p = xv >= tau ? ex2((xv - ms.x) * P.c) * invS : 0.0f;
      return qrow ? fmaxf(p - qv, 0.0f) : (v == excl ? 0.0f : p);
    };
    // f4(w[4], v): entries v .. v+3; f1(w, v): single entries of the remainder
    auto visit = [&](auto&& f4, auto&& f1) {
      int vs = v0;  // start of the scalar remainder
      if (P.vec_ok) {
        constexpr int kEl = 16 / sizeof(TT);
        const int n_vec = (v1 - v0) / kEl;
        const uint4* rv = reinterpret_cast<const uint4*>(row + v0);
        for (int j = threadIdx.x; j < n_vec; j += blockDim.x) {
          float x[kEl];
          unpack16<TT>(__ldg(rv + j), x);
          const int v = v0 + j * kEl;
#pragma unroll
          for (int h = 0; h < kEl / 4; ++h) {
            float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (qrow) q4 = __ldg(reinterpret_cast<const float4*>(qrow + v) + h);
            const float w[4] = {weight(x[4 * h + 0], q4.x, v + 4 * h + 0),
                                weight(x[4 * h + 1], q4.y, v + 4 * h + 1),
                                weight(x[4 * h + 2], q4.z, v + 4 * h + 2),
                                weight(x[4 * h + 3], q4.w, v + 4 * h + 3)};
            f4(w, v + 4 * h);
          }
        }
        vs = v0 + n_vec * kEl;
      }
      for (int v = vs + threadIdx.x; v < v1; v += blockDim.x)
        f1(weight(load_logit(row + v), qrow ? __ldg(qrow + v) : 0.0f, v), v);
    };
    // Seed: the slice's heaviest entry enters the race first, so that the
    // pruning in race_offer drops the log (and often the hash) of nearly every
    // other entry.  Pruning never changes the winner.
    float wmax = 0.0f;
    int imax = 0x7FFFFFFF;
    auto track = [&](float w, int v) {
      if (w > wmax || (w == wmax && w > 0.0f && v < imax)) {
        wmax = w;
        imax = v;
      }
    };
    visit([&](const float* w, int v) {
#pragma unroll
      for (int i = 0; i < 4; ++i) track(w[i], v + i);
    }, track);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float w2 = __shfl_xor_sync(0xFFFFFFFFu, wmax, o);
      const int i2 = __shfl_xor_sync(0xFFFFFFFFu, imax, o);
      if (w2 > wmax || (w2 == wmax && i2 < imax)) {
        wmax = w2;
        imax = i2;
      }
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float4(wmax, __int_as_float(imax), 0.f, 0.f);
    __syncthreads();
    Race best = race_none();
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      const float w2 = red[w].x;
      const int i2 = __float_as_int(red[w].y);
      if (w2 > wmax || (w2 == wmax && i2 < imax)) {
        wmax = w2;
        imax = i2;
      }
    }
    __syncthreads();
    if (wmax > 0.0f) race_offer(best, wmax, rkey, (uint32_t)imax);
    visit([&](const float* w, int v) { race_offer4(best, w, rkey, (uint32_t)v); },
          [&](float w, int v) { race_offer(best, w, rkey, (uint32_t)v); });
    const Race tb = block_race<TT>(best, red);
    if (threadIdx.x == 0) {
      P.rpart[(int64_t)k * P.rstride + sl] = make_float4(tb.w, tb.e, __int_as_float(tb.idx), 0.f);
      __threadfence();
      s_last = (atomicAdd(P.rcount + k, 1) == S - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      Race all = race_none();
      for (int s2 = 0; s2 < S; ++s2) {
        const float4 r = __ldcg(P.rpart + (int64_t)k * P.rstride + s2);
        race_merge(all, r.x, r.y, __float_as_int(r.z));
      }
      if (!(all.w > 0.0f)) {  // empty residual: race over p instead
        Race bp = race_none();
        for (int v = threadIdx.x; v < V; v += blockDim.x) {
          const float xv = load_logit(row + v);
          race_offer(bp, xv >= tau ? ex2((xv - ms.x) * P.c) * invS : 0.0f, rkey, (uint32_t)v);
        }
        all = block_race<TT>(bp, red);
      }
      if (threadIdx.x == 0) {
        P.out_tokens[t] = all.idx;
        P.rcount[k] = 0;
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Greedy path (T == 0).
// ---------------------------------------------------------------------------
// Argmax of every target row.  Work items are (row, chunk) pairs, a chunk being
// 256 vectors of 16 bytes (or 256 elements when rows are not 16-byte aligned);
// each warp takes items in grid-stride order, keeps 8 loads per lane in flight,
// reduces the packed (value, -index) keys over the warp and folds its result
// into the row's key with one 64-bit atomicMax.  No block-level barrier.  The
// finalize kernel reads the row keys and resets them to 0 for the next call.
template <typename TT>
__global__ void __launch_bounds__(kRowThreads) greedy_partial_kernel(const Params P, int vec_ok) {
  constexpr int kEl = 16 / sizeof(TT);
  constexpr int kPer = 8;                 // loads per lane per item
  constexpr int kChunkVec = 32 * kPer;    // vectors (or elements) per item
  const int B = P.B, V = P.V;
  const int64_t n_t = min((int64_t)__ldg(P.cu + B) + B, P.cap_rows);
  if (blockIdx.x == 0 && threadIdx.x == 0 && (int64_t)__ldg(P.cu + B) + B > P.cap_rows)
    set_err(P.err, SPECDEC_DEVERR_CAPACITY);
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int per_row = vec_ok ? (V / kEl + kChunkVec - 1) / kChunkVec : (V + kChunkVec - 1) / kChunkVec;
  const int64_t items = n_t * per_row;
  for (int64_t it = warp_id; it < items; it += nwarps) {
    const int64_t t = it / per_row;
    const int ch = (int)(it % per_row);
    const TT* row = reinterpret_cast<const TT*>(P.logits) + t * (int64_t)V;
    // The chunk's loads go out first (row t < cu[B] + B exists by the layout);
    // the request lookup (a binary search over cu) runs while they are in flight.
    const int nv = V / kEl;
    const int j0 = ch * kChunkVec + lane;
    uint4 w[kPer];
    if (vec_ok) {
#pragma unroll
      for (int k = 0; k < kPer; ++k)
        if (j0 + 32 * k < nv) w[k] = __ldg(reinterpret_cast<const uint4*>(row) + j0 + 32 * k);
    }
    // only rows of well-formed requests are accumulated: exactly the rows the
    // finalize kernel reads and resets
    const int b = request_of_target(P.cu, B, t);
    const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
    const int64_t t0 = (int64_t)c0 + b;
    if (g < 0 || t < t0 || t > t0 + g || t0 + g >= P.cap_rows) continue;
    // Each lane scans its elements in increasing index order, so a strict
    // "greater" keeps the lowest index on ties (and -0.0 == +0.0, as numbers).
    float bv = -INFINITY;
    int bi = -1;
    if (vec_ok) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int j = j0 + 32 * k;
        if (j >= nv) break;
        float x[kEl];
        unpack16<TT>(w[k], x);
#pragma unroll
        for (int h = 0; h < kEl; ++h)
          if (x[h] > bv || bi < 0) {
            bv = x[h];
            bi = j * kEl + h;
          }
      }
    } else {
      const int v0 = ch * kChunkVec + lane;
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int v = v0 + 32 * k;
        if (v < V) {
          const float x = load_logit(row + v);
          if (x > bv || bi < 0) {
            bv = x;
            bi = v;
          }
        }
      }
    }
    uint64_t best = bi < 0 ? 0ull : argmax_key(bv, (uint32_t)bi);
    best = warp_max_u64(best);
    if (lane == 0) atomicMax(reinterpret_cast<unsigned long long*>(P.gkeys + t), (unsigned long long)best);
  }
}

// One warp per request: lanes combine the partial argmax keys of the request's
// rows (lowest index on ties is built into the keys), lane 0 scans.
static __global__ void greedy_finalize_kernel(const Params P) {
  __shared__ int s_g[8][33];
  wait_for_previous_kernel();
  const int B = P.B, V = P.V;
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  for (int b = blockIdx.x * 8 + wib; b < B; b += gridDim.x * 8) {
    const int c0 = __ldg(P.cu + b), g = __ldg(P.cu + b + 1) - c0;
    const int64_t t0 = (int64_t)c0 + b;
    if (g < 0 || t0 + g >= P.cap_rows) continue;
    int n = g, tok = -1;
    bool found = false;
    // rows in chunks of 32 (row = chunk base + lane); every position's outputs
    // are written, also after the first rejection
    for (int i0 = 0; i0 <= g; i0 += 32) {
      const int i = i0 + lane;
      int gi = -1;
      if (i <= g) {
        gi = (int)argmax_key_index(P.gkeys[t0 + i]);
        P.gkeys[t0 + i] = 0;  // ready for the next call
      }
      s_g[wib][lane] = gi;
      int acc = 0;
      if (i < g) {
        const int x = __ldg(P.ids + c0 + i);
        if (x < 0 || x >= V) set_err(P.err, SPECDEC_DEVERR_BAD_DRAFT_ID);
        acc = (x == gi);
        const int64_t d = (int64_t)c0 + i;
        if (P.out_beta) P.out_beta[d] = acc ? 1.0f : 0.0f;
        if (P.out_px) P.out_px[d] = acc ? 1.0f : 0.0f;
        if (P.out_qx) P.out_qx[d] = 1.0f;
        if (P.out_acc) P.out_acc[d] = acc;
      }
      __syncwarp();
      // first rejected draft in this chunk (the bonus slot i == g counts as the stop)
      const unsigned stop = __ballot_sync(0xFFFFFFFFu, (i < g && !acc) || i == g);
      if (stop && !found) {
        const int f = __ffs(stop) - 1;
        n = i0 + f;
        tok = s_g[wib][f];
        found = true;
      }
      __syncwarp();
    }
    if (lane == 0) P.out_nacc[b] = n;
    for (int i = lane; i <= g; i += 32)
      P.out_tokens[t0 + i] = i < n ? __ldg(P.ids + c0 + i) : (i == n ? tok : -1);
  }
}

static __global__ void uniform_fill_kernel(uint64_t key, uint64_t v0, int64_t n, float* out) {
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
       j += (int64_t)gridDim.x * blockDim.x)
    out[j] = uniform_from_bits(uniform_bits(key, v0 + (uint64_t)j));
}

// -E = ln U for U(k) with k given: used by the tests of the log evaluation.
static __global__ void neglog_fill_kernel(uint32_t k0, int64_t n, float* out) {
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
       j += (int64_t)gridDim.x * blockDim.x)
    out[j] = neg_log_uniform(k0 + (uint32_t)j);
}

// The selection's integer mass and 2^-z of entries at distances z from the
// row maximum, for a row of V entries: used by the tests of the mass definition.
static __global__ void selection_mass_kernel(const float* z, int64_t n, int V,
                                             unsigned long long* mass, float* p2) {
  const float fscale = adj_mass_scale(adj_mass_shift(V));
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n;
       j += (int64_t)gridDim.x * blockDim.x) {
    const float zj = z[j];
    if (mass) mass[j] = adj_mass(zj, fscale);
    if (p2) p2[j] = pow2_neg(zj);
  }
}

}  // namespace specdec
