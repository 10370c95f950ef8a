// Device-side building blocks shared by the verifier kernels: the counter-based
// generator, the exponential-race key, numeric helpers and thin inline-PTX
// wrappers for mbarriers, bulk (TMA) copies and distributed shared memory.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/specdec.h"

namespace specdec {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Counter-based generator.  SplitMix64 (Steele, Lea, Flood, OOPSLA 2014): add
// the golden gamma, then the two xor-shift-multiply rounds and a final
// xor-shift.  The key chain and the 23-bit uniform are this library's own
// definition, documented in specdec.h.
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ uint64_t stream_key(uint64_t seed, uint64_t b, uint64_t pos,
                                                        uint64_t stream) {
  return splitmix64(splitmix64(splitmix64(seed) ^ b) ^ ((pos << 8) | stream));
}

// 23 bits for entry v: one hash of (key ^ (v >> 1)) serves the pair (2j, 2j+1),
// bits [41, 64) for even v and bits [18, 41) for odd v; U = (k + 1/2) 2^-23,
// k in [0, 2^23).
__device__ __forceinline__ uint32_t uniform_bits(uint64_t key, uint64_t v) {
  const uint64_t h = splitmix64(key ^ (v >> 1));
  return (v & 1) ? (uint32_t)(h >> 18) & 0x7FFFFFu : (uint32_t)(h >> 41);
}
// Both uniforms of the pair (2j, 2j + 1) from their one hash.
__device__ __forceinline__ void uniform_bits2(uint64_t key, uint64_t j, uint32_t& k0, uint32_t& k1) {
  const uint64_t h = splitmix64(key ^ j);
  k0 = (uint32_t)(h >> 41);
  k1 = (uint32_t)(h >> 18) & 0x7FFFFFu;
}

__device__ __forceinline__ float uniform_from_bits(uint32_t k) {
  // k < 2^23, so k + 0.5 has at most 24 significant bits: both steps are exact.
  return ((float)k + 0.5f) * (1.0f / 8388608.0f);
}

// E = -ln U for U = (k + 1/2) 2^-23, with small relative error over the whole
// range, branch-free.  Below U = 1/2 the hardware base-2 logarithm has a
// relative error of a few 2^-23 (|log2 U| >= 1).  Above it, d = 1 - U =
// (2^24 - 2k - 1) 2^-24 is exact and -ln(1 - d) = 2 atanh(s) with
// s = d / (2 - d) <= 1/3, summed as the odd power series
// 2 (s + s^3/3 + s^5/5 + ...) to s^15 (truncation below (1/9)^8 / 17 ~ 1.4e-9
// relative).  Both branches are evaluated and one is selected, so a warp never
// diverges here.
__device__ __forceinline__ float neg_log_uniform(uint32_t k) {
  const float u = uniform_from_bits(k);
  float l2;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(u));
  const float lo = -l2 * kLn2;
  const float d = (float)((1u << 24) - 2u * k - 1u) * (1.0f / 16777216.0f);
  const float s = __fdividef(d, 2.0f - d);
  const float s2 = s * s;
  float t = 1.0f / 15.0f;
  t = fmaf(t, s2, 1.0f / 13.0f);
  t = fmaf(t, s2, 1.0f / 11.0f);
  t = fmaf(t, s2, 1.0f / 9.0f);
  t = fmaf(t, s2, 1.0f / 7.0f);
  t = fmaf(t, s2, 1.0f / 5.0f);
  t = fmaf(t, s2, 1.0f / 3.0f);
  t = fmaf(t, s2, 1.0f);
  const float hi = 2.0f * s * t;
  return k < (1u << 22) ? lo : hi;
}

// Candidate of the exponential race: key w / e (larger wins), kept as the pair
// so that comparing two candidates needs two multiplies instead of a division
// per vocabulary entry.  w <= 0 means "no candidate".  Equal keys go to the
// lower vocabulary index, as in the oracle's ascending scan.
struct Race {
  float w;
  float e;
  int32_t idx;
};

__device__ __forceinline__ Race race_none() { return Race{0.0f, 1.0f, 0x7FFFFFFF}; }

__device__ __forceinline__ bool race_beats(float aw, float ae, int32_t ai, const Race& b) {
  if (!(aw > 0.0f)) return false;
  if (!(b.w > 0.0f)) return true;
  const float l = aw * b.e, r = b.w * ae;
  return l > r || (l == r && ai < b.idx);
}

__device__ __forceinline__ void race_merge(Race& a, float bw, float be, int32_t bi) {
  if (race_beats(bw, be, bi, a)) {
    a.w = bw;
    a.e = be;
    a.idx = bi;
  }
}

// Pruning that never changes the winner: E = -ln U >= 1 - U = d for every
// U, and d >= 2^-24 here, so an entry whose key bound w / d (computed with a
// 2^-16 margin, far above the rounding of the products) stays below the
// current best key a.w / a.e loses to it, and neither its log nor (when even
// d = 2^-24 cannot help) its hash is needed.
constexpr float kRaceMargin = 1.0f - 1.0f / 65536.0f;
__device__ __forceinline__ bool race_hopeless(const Race& a, float w, float d) {
  return a.w > 0.0f && w * a.e < a.w * (d * kRaceMargin);
}
__device__ __forceinline__ float one_minus_uniform(uint32_t k) {
  return (float)((1u << 24) - 2u * k - 1u) * (1.0f / 16777216.0f);  // exact
}

// Offers entries v .. v+3 with weights w[0..3]: the hashes are independent
// (no branch between them); only entries that pass the bound take the log and
// the comparison.  Checking all four against the best from before the group is
// conservative, so the result is the one race_offer gives one by one.
__device__ __forceinline__ void race_offer4(Race& a, const float* w, uint64_t key, uint32_t v) {
  uint32_t k[4];
  if ((v & 1u) == 0u) {  // two pairs: two hashes (every caller's v is a multiple of 4)
    uniform_bits2(key, v >> 1, k[0], k[1]);
    uniform_bits2(key, (v >> 1) + 1, k[2], k[3]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) k[i] = uniform_bits(key, v + i);
  }
  bool c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = w[i] > 0.0f && !race_hopeless(a, w[i], one_minus_uniform(k[i]));
  if (c[0] | c[1] | c[2] | c[3]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (c[i]) race_merge(a, w[i], neg_log_uniform(k[i]), (int32_t)(v + i));
  }
}

// Offers vocabulary entry v with weight w (w <= 0: not a candidate).
__device__ __forceinline__ void race_offer(Race& a, float w, uint64_t key, uint32_t v) {
  if (!(w > 0.0f) || race_hopeless(a, w, 1.0f / 16777216.0f)) return;
  const uint32_t k = uniform_bits(key, v);
  if (race_hopeless(a, w, one_minus_uniform(k))) return;
  race_merge(a, w, neg_log_uniform(k), (int32_t)v);
}

// exp2 on the special-function unit (flush-to-zero; arguments here are <= 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Online softmax state (m, s): s = sum exp2((x - m) * c) over the values seen.
__device__ __forceinline__ void softmax_merge(float& m, float& s, float m2, float s2, float c) {
  float mn = fmaxf(m, m2);
  if (mn == -INFINITY) {  // both empty or all -inf
    m = mn;
    s = 0.0f;
    return;
  }
  s = s * ex2((m - mn) * c) + s2 * ex2((m2 - mn) * c);
  m = mn;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename TT>
__device__ __forceinline__ float load_logit(const TT* p);
template <>
__device__ __forceinline__ float load_logit<float>(const float* p) {
  return __ldg(p);
}
template <>
__device__ __forceinline__ float load_logit<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p)) << 16);
}

// Ordered 64-bit key of (value, index) for argmax with the lowest index on ties:
// larger key = larger value, then smaller index.  -0.0 is folded into +0.0 so
// the two compare equal, as they do as numbers.
__device__ __forceinline__ uint64_t argmax_key(float x, uint32_t idx) {
  x = x + 0.0f;
  uint32_t b = __float_as_uint(x);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((uint64_t)b << 32) | (uint64_t)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t argmax_key_index(uint64_t k) {
  return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFu);
}

// Accept test r < min(1, p/q) with the conventions p = 0 -> reject,
// q = 0 < p -> accept.  r < 1 always, so min(1, .) needs no separate branch.
__device__ __forceinline__ bool accept_test(float r, float px, float qx) {
  if (!(px > 0.0f)) return false;
  if (!(qx > 0.0f)) return true;
  return r < __fdiv_rn(px, qx);
}

// Per-row status word written by the row kernels, read by later rows of the
// same request (inside the same launch) and by the finalize kernel:
// bits 63..8 = call epoch, bits 7..0 = flags.
constexpr uint32_t kStDone = 1u;
constexpr uint32_t kStAccepted = 2u;
constexpr uint32_t kStRaceDone = 4u;

__device__ __forceinline__ uint64_t make_status(uint64_t epoch, uint32_t flags) {
  return (epoch << 8) | (uint64_t)flags;
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Prefix state of a request before position i, from the status words of its
// earlier rows: 1 = all accepted, 2 = some rejected, 0 = not known yet.
constexpr int kPrefixUnknown = 0;
constexpr int kPrefixAllAccepted = 1;
constexpr int kPrefixRejected = 2;

// The status words are read eight at a time, all loads issued before any is
// looked at, so a prefix of i positions costs about ceil(i / 8) load latencies
// (the thread that takes a work slot waits on this while its CTA idles).
__device__ __forceinline__ int read_prefix(const uint64_t* status, int64_t t_first, int i,
                                           uint64_t epoch) {
  int state = kPrefixAllAccepted;
  for (int j0 = 0; j0 < i; j0 += 8) {
    uint64_t s[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = j0 + j < i ? ld_relaxed_u64(status + t_first + j0 + j) : 0ull;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j0 + j >= i) break;
      if ((s[j] >> 8) != epoch || !(s[j] & kStDone)) {
        state = kPrefixUnknown;
        continue;
      }
      if (!(s[j] & kStAccepted)) return kPrefixRejected;
    }
  }
  return state;
}

// Request index of draft position d: the b with cu[b] <= d < cu[b+1]
// (first b whose cu[b+1] > d; empty requests are skipped).
__device__ __forceinline__ int request_of_draft(const int32_t* cu, int B, int64_t d) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if ((int64_t)__ldg(cu + mid + 1) > d)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo;
}
// Request index of target row t: the b with cu[b] + b <= t <= cu[b+1] + b.
__device__ __forceinline__ int request_of_target(const int32_t* cu, int B, int64_t t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if ((int64_t)__ldg(cu + mid + 1) + mid + 1 > t)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier / bulk copy / cluster wrappers (PTX ISA, sm_90+ forms).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster (address from mapa).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
// try_wait with a suspend-time hint: a thread whose phase is not complete sleeps
// in hardware until it completes (or the hint, 1 ms, runs out) instead of
// spinning and taking issue slots from the warps that do the work.
constexpr uint32_t kSuspendHintNs = 1000000u;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after `limit_ns` of wall time and returns false.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait_acq_cluster(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Bulk global -> shared copy completing on `bar` (bytes % 16 == 0, both
// addresses 16-byte aligned).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t ncluster_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c,
                                              float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Named barrier that also ORs a predicate over the participating threads, so
// every thread leaves with the same answer.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Warp reductions.
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}
__device__ __forceinline__ void warp_softmax(float& m, float& s, float c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    softmax_merge(m, s, m2, s2, c);
  }
}
__device__ __forceinline__ void warp_race(Race& r) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w2 = __shfl_xor_sync(0xFFFFFFFFu, r.w, o);
    const float e2 = __shfl_xor_sync(0xFFFFFFFFu, r.e, o);
    const int32_t i2 = __shfl_xor_sync(0xFFFFFFFFu, r.idx, o);
    race_merge(r, w2, e2, i2);
  }
}
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    uint64_t y = __shfl_xor_sync(0xFFFFFFFFu, x, o);
    x = y > x ? y : x;
  }
  return x;
}

}  // namespace specdec
