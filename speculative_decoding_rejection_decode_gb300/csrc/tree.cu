// Token-tree verification: several draft candidates per position.
//
// The tree drafts that the tarrragon page names (EAGLE) give a node several
// children: candidates for the same next token, each drawn independently from
// that node's draft distribution q_u.  The pages state the accept rule for one
// candidate per position only (the vllbc page, Section 3.6, notes that any
// drafter works as long as its probabilities are known at verification).  This
// library repeats that rule after each rejection, with the normalised residual
// as the next candidate's target, which the correctness argument of the vllbc
// page's Appendix A.1 covers at every round:
//   at node u with target t (first the softmax p_u of target row u),
//   candidate r (the r-th child, in node order) with token x is accepted when
//   U(seed, b, u, 0, r) < min(1, t(x) / q_u(x)); otherwise t <- norm(max(0,
//   t - q_u)) (t unchanged if that is zero everywhere).  An accepted candidate
//   becomes the next node; after the last rejection, or at a node without
//   children, the extra token is drawn from t by the exponential race with the
//   uniforms U(seed, b, u, 1, v).
// On a chain this is exactly the chain verifier.
//
// Every target after r rejections has the closed form
//     t_r(v) = max(0, p(v) - C_r q(v)) / D_r,   C_0 = 0, D_0 = 1,
//     C_{r+1} = C_r + D_r,  D_{r+1} = sum_v max(0, p(v) - C_{r+1} q(v)),
// so the kernel keeps two scalars per round and needs one pass over the
// (target, draft) row pair for each rejection that is followed by another
// candidate, plus one for the race.
//
// One CTA walks one request at a time (requests taken from a counter): per
// visited node a pass for (max, sum) of the target row, the accept tests (one
// gather each), the residual passes and the race.  Only the rows of visited
// nodes are read.
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "tree.cuh"

namespace specdec {

namespace {


// Sum over the row pair of w(v) = max(0, p(v) - C q(v)) (w = p without q),
// p(v) = 2^((l_v - M) c) / S, and, with kRace, the race over w with key rkey.
// Per-thread partial sum and race candidate (reduced by the caller).
template <typename TT, int NT, bool kHasQ, bool kRace>
__device__ __forceinline__ void tree_pass(const TT* row, const float* qrow, int V, bool vec,
                                          float M, float c, float invS, float C, uint64_t rkey,
                                          uint64_t pol, float& wsum, Race& best) {
  constexpr int kEl = 16 / sizeof(TT);
  const int tid = threadIdx.x;
  auto four = [&](const float* l, const float4& q4, uint32_t v) {
    const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
    float w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float p = ex2((l[k] - M) * c) * invS;
      w[k] = kHasQ ? fmaxf(p - C * qv[k], 0.0f) : p;
    }
    wsum += (w[0] + w[1]) + (w[2] + w[3]);
    if constexpr (kRace) {
      if ((w[0] > 0.0f) | (w[1] > 0.0f) | (w[2] > 0.0f) | (w[3] > 0.0f)) race_offer4(best, w, rkey, v);
    }
  };
  if (vec) {
    const uint4* rv = reinterpret_cast<const uint4*>(row);
    const uint4* qv = reinterpret_cast<const uint4*>(qrow);
    const int nv = V / kEl;
    // U vectors (and their draft entries) in flight per thread, then the tail
    constexpr int U = kRace ? 2 : 4;
    int j = tid;
    for (; j + (U - 1) * NT < nv; j += U * NT) {
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
          float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
          if constexpr (kHasQ) q4 = *reinterpret_cast<const float4*>(&b[u][h]);
          four(x + 4 * h, q4, (uint32_t)((j + u * NT) * kEl + 4 * h));
        }
      }
    }
    for (; j < nv; j += NT) {
      float x[kEl];
      unpack16<TT>(ldg_hint(rv + j, pol), x);
#pragma unroll
      for (int h = 0; h < kEl / 4; ++h) {
        float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (kHasQ) {
          const uint4 b = ldg_hint(qv + j * (kEl / 4) + h, pol);
          q4 = *reinterpret_cast<const float4*>(&b);
        }
        four(x + 4 * h, q4, (uint32_t)(j * kEl + 4 * h));
      }
    }
  } else {
    for (int v = tid; v < V; v += NT) {
      const float p = ex2((load_logit(row + v) - M) * c) * invS;
      const float w = kHasQ ? fmaxf(p - C * __ldg(qrow + v), 0.0f) : p;
      wsum += w;
      if constexpr (kRace) race_offer(best, w, rkey, (uint32_t)v);
    }
  }
}

// Block-wide sum and race merge (every thread gets both); ends on a barrier.
template <int NT>
__device__ __forceinline__ void tree_reduce(float& wsum, Race& best, float4* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  wsum = warp_sum(wsum);
  warp_race(best);
  __syncthreads();  // red may still be read from the previous reduction
  if (lane == 0) red[warp] = make_float4(wsum, best.w, best.e, __int_as_float(best.idx));
  __syncthreads();
  float s = 0.0f;
  Race r = race_none();
  for (int w = 0; w < (NT / 32); ++w) {
    s += red[w].x;
    race_merge(r, red[w].y, red[w].z, __float_as_int(red[w].w));
  }
  wsum = s;
  best = r;
}

template <typename TT, int NT, int MINB>
__global__ void __launch_bounds__(NT, MINB) tree_walk_kernel(const TreeArgs P) {
  constexpr int kTreeThreads = NT, kTreeWarps = NT / 32;
  __shared__ float4 red[kTreeWarps];
  __shared__ unsigned long long s_key[kTreeWarps];
  __shared__ int s_cnt[kTreeWarps];
  __shared__ int s_ch[kTreeMaxChildren];
  __shared__ int s_req, s_nch, s_bad, s_acc;
  constexpr int kEl = 16 / sizeof(TT);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = P.V;
  const bool vec = P.vec_ok != 0;
  const bool greedy = P.c == 0.0f;
  const uint64_t keep = policy_evict_last(), drop = policy_evict_first();

  for (;;) {
    if (tid == 0) {
      const unsigned long long k = atomicAdd(P.counter, 1ull);
      s_req = k < (unsigned long long)P.B ? (int)k : -1;
      s_bad = 0;
    }
    __syncthreads();
    const int b = s_req;
    if (b < 0) break;
    const int64_t n0 = __ldg(P.cu + b);
    const int n = __ldg(P.cu + b + 1) - (int)n0;
    // the request's tree: node 0 first, every other node after its parent
    {
      int bad = (n < 1 || (b == 0 && n0 != 0)) ? 1 : 0;
      for (int j = tid; j < n && !bad; j += kTreeThreads) {
        const int pj = __ldg(P.par + n0 + j);
        bad = j == 0 ? (pj != -1) : (pj < 0 || pj >= j);
      }
      if (bad) atomicOr(&s_bad, 1);
    }
    __syncthreads();
    if (s_bad) {
      if (tid == 0) set_err(P.err, n < 1 || (b == 0 && n0 != 0) ? SPECDEC_DEVERR_BAD_CU
                                                                 : SPECDEC_DEVERR_BAD_TREE);
      __syncthreads();
      continue;
    }
    const uint64_t gen = P.req_offset + (uint64_t)b;
    int u = 0, depth = 0, extra = -1;
    for (;;) {
      const TT* row = reinterpret_cast<const TT*>(P.logits) + (n0 + u) * (int64_t)V;
      const float* qrow = greedy ? nullptr : P.q + (n0 + u) * (int64_t)V;
      // ---- the children of u, in node order (an ordered compaction) -------
      if (tid == 0) s_nch = 0;
      __syncthreads();
      for (int j0 = u + 1; j0 < n; j0 += kTreeThreads) {
        const int j = j0 + tid;
        const bool f = j < n && __ldg(P.par + n0 + j) == u;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, f);
        if (lane == 0) s_cnt[warp] = __popc(m);
        __syncthreads();
        int off = s_nch;
        for (int w = 0; w < warp; ++w) off += s_cnt[w];
        off += __popc(m & ((1u << lane) - 1u));
        if (f && off < kTreeMaxChildren) s_ch[off] = j;
        __syncthreads();
        if (tid == 0) {
          int tot = 0;
          for (int w = 0; w < kTreeWarps; ++w) tot += s_cnt[w];
          s_nch += tot;
        }
        __syncthreads();
      }
      const int nch = s_nch;
      if (nch > kTreeMaxChildren && tid == 0) set_err(P.err, SPECDEC_DEVERR_CAPACITY);
      const int K = min(nch, kTreeMaxChildren);
      int next = -1;

      if (greedy) {
        // ---- T == 0: the argmax of the row (lowest index on ties) ------------
        uint64_t best = 0ull;
        if (vec) {
          const uint4* rv = reinterpret_cast<const uint4*>(row);
          for (int j = tid; j < V / kEl; j += kTreeThreads) {
            float x[kEl];
            unpack16<TT>(ldg_hint(rv + j, drop), x);
#pragma unroll
            for (int e = 0; e < kEl; ++e) {
              const uint64_t k = argmax_key(x[e], (uint32_t)(j * kEl + e));
              best = k > best ? k : best;
            }
          }
        } else {
          for (int v = tid; v < V; v += kTreeThreads) {
            const uint64_t k = argmax_key(load_logit(row + v), (uint32_t)v);
            best = k > best ? k : best;
          }
        }
        best = warp_max_u64(best);
        if (lane == 0) s_key[warp] = best;
        __syncthreads();
        uint64_t g = 0ull;
        for (int w = 0; w < kTreeWarps; ++w) g = s_key[w] > g ? s_key[w] : g;
        const int gi = (int)argmax_key_index(g);
        if (tid == 0) {
          int nx = -1;
          for (int r = 0; r < K; ++r) {
            const int x = __ldg(P.tok + n0 + s_ch[r]);
            if (x < 0 || x >= V) set_err(P.err, SPECDEC_DEVERR_BAD_DRAFT_ID);
            if (x == gi) {
              nx = s_ch[r];
              break;
            }
          }
          s_acc = nx;
        }
        __syncthreads();
        next = s_acc;
        extra = gi;
      } else {
        // ---- T > 0: (max, sum) of the target row ----------------------------
        const int hi = vec ? V / kEl : V;
        float m0, s0;
        sweep1<TT, kTreeThreads>(row, 0, hi, vec, P.c, keep, m0, s0);
        warp_softmax(m0, s0, P.c);
        __syncthreads();
        if (lane == 0) red[warp] = make_float4(m0, s0, 0.f, 0.f);
        __syncthreads();
        float M = -INFINITY, S = 0.0f;
        for (int w = 0; w < kTreeWarps; ++w) softmax_merge(M, S, red[w].x, red[w].y, P.c);
        const float invS = 1.0f / S;
        // ---- candidates in order; the target is max(0, p - C q) / D ---------
        float C = 0.0f, D = 1.0f;
        for (int r = 0; r < K; ++r) {
          if (tid == 0) {
            const int x = __ldg(P.tok + n0 + s_ch[r]);
            float cur = 0.0f, qx = 0.0f;
            if (x >= 0 && x < V) {
              const float px = ex2((load_logit(row + x) - M) * P.c) * invS;
              qx = __ldg(qrow + x);
              cur = fmaxf(px - C * qx, 0.0f) / D;
            } else {
              set_err(P.err, SPECDEC_DEVERR_BAD_DRAFT_ID);
            }
            const float rr = uniform_from_bits(uniform_bits(stream_key(P.seed, gen, u, 0), r));
            s_acc = accept_test(rr, cur, qx) ? 1 : 0;
          }
          __syncthreads();
          const bool acc = s_acc != 0;
          __syncthreads();  // s_acc is rewritten in the next round
          if (acc) {
            next = s_ch[r];
            break;
          }
          if (r + 1 < K) {
            // the residual the next candidate is tested against
            float W = 0.0f;
            Race none = race_none();
            tree_pass<TT, NT, true, false>(row, qrow, V, vec, M, P.c, invS, C + D, 0ull, drop, W, none);
            tree_reduce<NT>(W, none, red);
            if (W > 0.0f) {
              C += D;
              D = W;
            }
          }
        }
        if (next < 0) {
          // ---- the extra token: the race over the last target ----------------
          const uint64_t rkey = stream_key(P.seed, gen, u, 1);
          float W = 0.0f;
          Race best = race_none();
          if (K == 0) {
            tree_pass<TT, NT, false, true>(row, qrow, V, vec, M, P.c, invS, 0.0f, rkey, drop, W, best);
            tree_reduce<NT>(W, best, red);
          } else {
            tree_pass<TT, NT, true, true>(row, qrow, V, vec, M, P.c, invS, C + D, rkey, drop, W, best);
            tree_reduce<NT>(W, best, red);
            if (!(W > 0.0f)) {  // zero residual: the target stays the previous one
              W = 0.0f;
              best = race_none();
              if (C > 0.0f)
                tree_pass<TT, NT, true, true>(row, qrow, V, vec, M, P.c, invS, C, rkey, drop, W, best);
              else
                tree_pass<TT, NT, false, true>(row, qrow, V, vec, M, P.c, invS, 0.0f, rkey, drop, W,
                                           best);
              tree_reduce<NT>(W, best, red);
            }
          }
          extra = best.w > 0.0f ? best.idx : 0;
        }
      }
      // ---- emit -------------------------------------------------------------
      if (next >= 0) {
        if (tid == 0) {
          P.out_tokens[n0 + depth] = __ldg(P.tok + n0 + next);
          if (P.out_path) P.out_path[n0 + depth] = next;
        }
        ++depth;
        u = next;
        continue;
      }
      if (tid == 0) {
        P.out_tokens[n0 + depth] = extra;
        P.out_nacc[b] = depth;
      }
      for (int j = depth + 1 + tid; j < n; j += kTreeThreads) P.out_tokens[n0 + j] = -1;
      if (P.out_path)
        for (int j = depth + tid; j < n; j += kTreeThreads) P.out_path[n0 + j] = -1;
      break;
    }
    __syncthreads();
  }
}

}  // namespace

int launch_tree(const TreeArgs& a, int dtype, int num_sms, cudaStream_t st) {
  if (cudaMemsetAsync(a.counter, 0, sizeof(unsigned long long), st) != cudaSuccess)
    return SPECDEC_ERR_CUDA;
  constexpr int kThreads = 512, kPerSm = 2;
  const int grid = num_sms * kPerSm;
  if (dtype == SPECDEC_BF16)
    tree_walk_kernel<__nv_bfloat16, kThreads, kPerSm><<<grid, kThreads, 0, st>>>(a);
  else
    tree_walk_kernel<float, kThreads, kPerSm><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

}  // namespace specdec
