// dspark_verify.cu -- batched speculative verification on GB300 (sm_103a).
//
// Method: "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation", section 2.1 (ratio test min(1, p_t/p_d) at
// every draft position, scanned left to right, the first rejection ends the
// block), section 1 (one bonus token), Appendix 8 (a fresh token from p_t when
// nothing is admitted). The residual max(0, p_t - p_d) after a rejection is the
// standard rule of the speculative sampling papers cited there as [1], [2].
//
// Pipeline (launches on the caller's stream, no host synchronisation):
//   k_plan      one CTA: validates verify lengths and row offsets, lays out the
//               rows to read (l_r + 1 target rows and l_r draft rows per
//               request) and resets counters.
//   k_rowstats  the streaming pass, HBM-bound. Persistent grid of 16 warps per
//               SM; every warp is an independent streamer with its own ring of
//               shared-memory stages fed by 4 KB 1-D bulk copies (TMA). A work
//               unit is 16 KB of one row. Each lane keeps an integer exponent
//               reference K (about ceil(max z * c), c = log2(e)/T, raised only
//               when its data outgrow it, by exact power-of-two rescaling) and
//               accumulates 2^(z*c - K) -- two FMAs and one ex2 per logit -- as
//               pairwise sums with Kahan compensation across chunks. Lanes merge
//               by exact powers of two and a TwoSum reduction; the unit's
//               statistics (sum as a float pair, K) go to the workspace. No
//               double-precision instruction runs per logit: GB300's FP64 rate
//               is a small fraction of its FP32 rate.
//   k_desc      one CTA per request: loads the tested tokens' logits, merges the
//               unit records of the request's rows (contiguous; a few threads
//               per row, compensated float, exact power-of-two alignment),
//               evaluates p_t^k(x_k)/p_d^k(x_k) in float -- in double only when
//               the uniform lies within 2e-6 of it -- finds the first
//               rejection with a warp ballot, writes accepted lengths, tokens
//               and probabilities, and the descriptor of the token to draw.
//   k_resid     the residual (or bonus) weights of every draw, summed per
//               2048-token segment by a persistent streamer like k_rowstats:
//               each warp's TMA ring carries 2 KB of the target row and 2 KB
//               of the draft row per stage.
//   k_pick      one CTA per request: scans the segment sums, re-reads the one
//               segment holding the cut and picks the token.
// Rows that are not 16-byte aligned take k_rowstats_plain (plain loads) and
// k_decide (several CTAs per request: ratio tests, segment sums, the draw).
#include <cuda.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "dspark_common.cuh"
#include "dspark_rowstats.cuh"
#include "dspark_verify_types.cuh"

namespace dspark {

struct __align__(16) ResampleDesc {
  int64_t t_row;  // global row of the target distribution sampled from
  int64_t d_row;  // global draft row (residual mode)
  int32_t K_t;    // exponent reference of the target row
  float D_hi;     // residual: log2(p_t/p_d)(v) = (z_t - z_d)*c - D, D = D_hi + D_lo
  float D_lo;
  float u;        // resample uniform
  int32_t mode;   // 0 nothing to do, 1 residual, 2 target distribution
  int32_t m;      // accepted count: position of the sampled token
  float E_hi;     // residual: D - K_t = E_hi + E_lo, so that p_d/p_t = 2^(z_d*c + E) / e_t
  float E_lo;
  float S_hi;     // acceptance jobs: the target row's sum_v 2^(z_v*c - K_t)
  float S_lo;
  int32_t pad[2];
};
static_assert(sizeof(ResampleDesc) == 64, "ResampleDesc layout");

// kModeMin: the acceptance probability's sum_v min(e_t(v), e_d(v)) (a job of
// dspark_acceptance, not a draw)
enum { kModeNone = 0, kModeResidual = 1, kModeTarget = 2, kModeMin = 3 };

// ---------------------------------------------------------------------------
// k_plan
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_plan(const int32_t* __restrict__ verify_len,
                                               const int64_t* __restrict__ toff,
                                               const int64_t* __restrict__ doff, int B,
                                               int gamma, VerifyWs ws, uint32_t* ties,
                                               int32_t* status) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  __shared__ int32_t sh_start[1025];  // this chunk's row starts (and the chunk's end)
  __shared__ long long sh_tb[1024], sh_db[1024];  // this chunk's first target and draft rows
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    *status = DSPARK_OK;
    *ties = 0;
    ws.hdr->next_unit = 0ull;
    ws.hdr->next_item = 0ull;
    ws.hdr->next_rate = 0ull;
    carry = 0;
  }
  __syncthreads();
  for (int base = 0; base < B; base += 1024) {
    const int r = base + tid;
    int cnt = 0;
    if (r < B) {
      // the request's first rows, kept for the row list below (no dependent
      // load per request there)
      sh_tb[tid] = toff ? toff[r] : static_cast<long long>(r) * (gamma + 1);
      sh_db[tid] = doff ? doff[r] : static_cast<long long>(r) * gamma;
      const int ell = verify_len[r];
      bool ok = ell >= 0 && ell <= gamma;
      if (ok && toff) {
        // rows of a valid request stay inside [0, toff[B]) and [0, doff[B]), the row
        // counts of the buffers, whatever the offsets of other requests hold
        const long long t0 = toff[r], t1 = toff[r + 1], d0 = doff[r], d1 = doff[r + 1];
        ok = t0 >= 0 && d0 >= 0 && t1 - t0 >= ell + 1 && d1 - d0 >= ell && t1 <= toff[B] &&
             d1 <= doff[B];
      }
      if (ok)
        cnt = 2 * ell + 1;
      else
        set_status(status, DSPARK_ERR_BAD_DATA);
      ws.tickets[r] = 0;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, w, o);
        if (lane >= o) w += v;
      }
      warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    // (past the batch cnt = 0, so a thread's start is the chunk's end)
    const int before = carry + (warp ? warp_tot[warp - 1] : 0) + incl - cnt;
    if (r < B) ws.req_row_start[r] = before;
    sh_start[tid] = before;
    __syncthreads();
    if (tid == 0) {
      carry += warp_tot[31];
      sh_start[1024] = carry;
    }
    __syncthreads();
    // the chunk's row list: one warp per request, lanes over its rows
    // (coalesced stores), the starts and first rows from shared memory
    const int nb = B - base < 1024 ? B - base : 1024;
    for (int q = warp; q < nb; q += 32) {
      const int start = sh_start[q], end = sh_start[q + 1];
      if (end == start) continue;  // invalid request: nothing to read
      const int ell = (end - start - 1) / 2;
      const long long tb = sh_tb[q], db = sh_db[q];
      for (int i = lane; i < end - start; i += 32)
        ws.row_list[start + i] = i <= ell ? (tb + i) << 1 : ((db + i - ell - 1) << 1) | 1;
    }
    __syncthreads();  // sh_start is rewritten by the next chunk
  }
  if (tid == 0) {
    ws.req_row_start[B] = carry;
    ws.hdr->total_rows = carry;
  }
}

// ---------------------------------------------------------------------------
// k_verify: ratio tests and the first-reject scan
// ---------------------------------------------------------------------------
struct RowStat {
  float S_hi, S_lo;  // sum_v 2^(z_v*c - K)
  int32_t K;
  bool ok;
};

// 2^a for a double exponent: split into an integer and a fraction in
// [-0.5, 0.5] so that the float exponential only sees a small argument
// (relative error ~1 ulp whatever the size of a). A few double operations per
// call; used per tested position, never per logit.
__device__ __forceinline__ float exp2_split(double a) {
  if (!(a > -1.0e4)) return 0.f;
  const double n = rint(a);
  return ldexpf(exp2f(static_cast<float>(a - n)), static_cast<int>(fmin(n, 1.0e4)));
}

// log2(p(x)) + log2(S) + K = z*c, so p(x) = 2^(z*c - K) / S.
__device__ __forceinline__ float prob_f32(float z, const RowStat& s, const ExpParams& ep) {
  return exp2_split(static_cast<double>(z) * ep.c_d - static_cast<double>(s.K)) /
         (s.S_hi + s.S_lo);
}

__device__ __forceinline__ double prob_f64(float z, const RowStat& s, const ExpParams& ep) {
  const double a = static_cast<double>(z) * ep.c_d - static_cast<double>(s.K);
  return exp2(a) / (static_cast<double>(s.S_hi) + static_cast<double>(s.S_lo));
}

// (K, hi, lo) += (K2, h2, l2): align by an exact power of two, add by TwoSum.
__device__ __forceinline__ void stat_combine(int& K, float& hi, float& lo, int K2, float h2,
                                             float l2) {
  if (K2 == INT_MIN) return;
  if (K == INT_MIN) {
    K = K2;
    hi = h2;
    lo = l2;
    return;
  }
  if (K2 > K) {
    hi = scale_pow2(hi, K - K2);
    lo = scale_pow2(lo, K - K2);
    K = K2;
  } else {
    h2 = scale_pow2(h2, K2 - K);
    l2 = scale_pow2(l2, K2 - K);
  }
  two_sum_acc(hi, lo, h2, l2);
}

// Records written by other CTAs of the running grid are read through L2
// (ld.global.cg), never through the non-coherent read-only path.
template <typename T>
__device__ __forceinline__ T ld_record(const T* p) {
  static_assert(sizeof(T) % 16 == 0 && alignof(T) == 16, "16-byte records");
  T v;
  const int4* src = reinterpret_cast<const int4*>(p);
  int4* o = reinterpret_cast<int4*>(&v);
#pragma unroll
  for (int i = 0; i < static_cast<int>(sizeof(T) / 16); ++i) o[i] = __ldcg(src + i);
  return v;
}

// One row's statistics from its unit records, all lanes of a warp: lanes take
// units, then a butterfly combine. Lane 0's result is the one used.
__device__ RowStat warp_merge_row(const TileStat* __restrict__ t, int n_units, int lane) {
  int K = INT_MIN;
  float hi = 0.f, lo = 0.f;
  bool bad = false;
  for (int u = lane; u < n_units; u += 32) {
    const TileStat ts = t[u];
    bad = bad || ts.bad != 0;
    stat_combine(K, hi, lo, ts.K, ts.s_hi, ts.s_lo);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const int K2 = __shfl_xor_sync(0xFFFFFFFFu, K, o);
    const float h2 = __shfl_xor_sync(0xFFFFFFFFu, hi, o);
    const float l2 = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
    stat_combine(K, hi, lo, K2, h2, l2);
  }
  RowStat r;
  const float s = hi + lo;
  r.S_hi = s;
  r.S_lo = lo - (s - hi);
  r.K = K;
  r.ok = !__any_sync(0xFFFFFFFFu, bad) && K != INT_MIN && s > 0.f && isfinite(s);
  return r;
}

// The statistics of nrows consecutive rows (unit records from t0) into
// sh_rs[0 .. nrows), by the whole CTA: tpr threads per row, each combining
// every tpr-th unit (four records in flight), then a butterfly over the row's
// lanes.
__device__ void merge_rows_block(const TileStat* __restrict__ t0, int nrows, int n_units,
                                 RowStat* sh_rs) {
  const int tpr = nrows <= static_cast<int>(blockDim.x) / 8   ? 8
                  : nrows <= static_cast<int>(blockDim.x) / 4 ? 4
                                                              : 2;
  const int tid = threadIdx.x, sub = tid & (tpr - 1);
  const int per_pass = static_cast<int>(blockDim.x) / tpr;
  for (int base = 0; base < nrows; base += per_pass) {
    const int row = base + tid / tpr;
    int K = INT_MIN;
    float hi = 0.f, lo = 0.f;
    bool bad = false;
    if (row < nrows) {
      const TileStat* t = t0 + static_cast<long long>(row) * n_units;
      int u = sub;
      for (; u + 3 * tpr < n_units; u += 4 * tpr) {
        const TileStat b0 = t[u], b1 = t[u + tpr], b2 = t[u + 2 * tpr], b3 = t[u + 3 * tpr];
        bad = bad || (b0.bad | b1.bad | b2.bad | b3.bad) != 0;
        stat_combine(K, hi, lo, b0.K, b0.s_hi, b0.s_lo);
        stat_combine(K, hi, lo, b1.K, b1.s_hi, b1.s_lo);
        stat_combine(K, hi, lo, b2.K, b2.s_hi, b2.s_lo);
        stat_combine(K, hi, lo, b3.K, b3.s_hi, b3.s_lo);
      }
      for (; u < n_units; u += tpr) {
        const TileStat b = t[u];
        bad = bad || b.bad != 0;
        stat_combine(K, hi, lo, b.K, b.s_hi, b.s_lo);
      }
    }
    for (int o = tpr / 2; o > 0; o >>= 1) {  // lanes of a row are an aligned group
      const int K2 = __shfl_xor_sync(0xFFFFFFFFu, K, o);
      const float h2 = __shfl_xor_sync(0xFFFFFFFFu, hi, o);
      const float l2 = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
      bad = (__shfl_xor_sync(0xFFFFFFFFu, bad ? 1 : 0, o) != 0) || bad;
      stat_combine(K, hi, lo, K2, h2, l2);
    }
    if (row < nrows && sub == 0) {
      RowStat rs;
      const float sm = hi + lo;
      rs.S_hi = sm;
      rs.S_lo = lo - (sm - hi);
      rs.K = K;
      rs.ok = !bad && K != INT_MIN && sm > 0.f && isfinite(sm);
      sh_rs[row] = rs;
    }
  }
}

// Inputs of the ratio test at position k = lane + 1 (and, in lane 0, the
// uniform of the draw after the block). They do not depend on the row
// statistics, so they are loaded while those are merged.
struct RatioIn {
  int32_t x;      // draft token, clamped into [0, V)
  float u;        // its uniform
  float zt, zd;   // target and draft logits at x
  float u_draw;   // lane 0: the uniform of the token drawn after the block
  bool bad;       // token or uniform out of range
};

template <typename Tin>
__device__ __forceinline__ RatioIn load_ratio_inputs(const Tin* __restrict__ tl,
                                                     const Tin* __restrict__ dl,
                                                     const int32_t* __restrict__ tokens,
                                                     const float* __restrict__ uniforms, int r,
                                                     int gamma, int V, int start, int ell,
                                                     const VerifyWs& ws, int lane) {
  RatioIn in{0, 0.f, 0.f, 0.f, 0.f, false};
  const int k = lane + 1;
  if (lane == 0) in.u_draw = uniforms[static_cast<long long>(r) * (gamma + 1) + gamma];
  if (k <= ell) {
    int32_t x = tokens[static_cast<long long>(r) * gamma + k - 1];
    const float u = uniforms[static_cast<long long>(r) * (gamma + 1) + k - 1];
    in.bad = x < 0 || x >= V || !(u >= 0.f && u < 1.f);
    x = min(max(x, 0), V - 1);
    const long long trow = ws.row_list[start + k - 1] >> 1;
    const long long drow = ws.row_list[start + ell + k] >> 1;
    in.x = x;
    in.u = u;
    in.zt = to_float<Tin>(tl[trow * V + x]);
    in.zd = to_float<Tin>(dl[drow * V + x]);
  }
  return in;
}

// Ratio tests of request r by one warp (lane k-1 tests position k), from the
// row statistics in sh_rs (target rows 0..ell, draft rows ell+1..2ell). With
// write_out it stores accepted_len, the accepted tokens, the probabilities and
// the near ties of these decisions. Lane 0 writes the descriptor of the token
// to draw after the block to *d_out.
template <typename Tin>
__device__ void ratio_tests(const RatioIn& in, int r, int gamma, int start, const RowStat* sh_rs,
                            const ExpParams& ep, const VerifyWs& ws, bool write_out,
                            int32_t* __restrict__ accepted_len, int32_t* __restrict__ emitted,
                            float* __restrict__ probs_out, uint32_t* ties, int32_t* status,
                            ResampleDesc* d_out, int lane, int end) {
  int32_t* em = emitted + static_cast<long long>(r) * (gamma + 1);
  float* pr = probs_out ? probs_out + static_cast<long long>(r) * gamma * 2 : nullptr;
  const int ell = (end - start - 1) / 2;
  const int k = lane + 1;  // the position this lane tests
  const bool has = k <= ell;
  float pt = 0.f, pd = 1.f;
  bool accept = false, tie = false;
  int32_t x = 0;
  RowStat st{}, sd{};
  double Dk = 0.0;  // this position's D, should it be the first rejection
  if (has) {
    st = sh_rs[k - 1];
    sd = sh_rs[ell + k];
    // independent of the ratio below: its latency overlaps the test's
    Dk = static_cast<double>(st.K - sd.K) +
         log2((static_cast<double>(st.S_hi) + st.S_lo) / (static_cast<double>(sd.S_hi) + sd.S_lo));
    x = in.x;
    const float u = in.u;
    if (in.bad || !st.ok || !sd.ok) set_status(status, DSPARK_ERR_BAD_DATA);
    const float zt = in.zt, zd = in.zd;
    pt = prob_f32(zt, st, ep);
    pd = prob_f32(zd, sd, ep);
    // ratio = 2^((z_t - z_d)*c - (K_t - K_d)) * S_d / S_t (relative error a few 1e-7)
    const double a = (static_cast<double>(zt) - static_cast<double>(zd)) * ep.c_d -
                     static_cast<double>(st.K - sd.K);
    const float ratio32 = exp2_split(a) * ((sd.S_hi + sd.S_lo) / (st.S_hi + st.S_lo));
    if (fabsf(u - ratio32) > 2e-6f && isfinite(ratio32)) {
      accept = u < ratio32;
    } else {  // close call: decide and flag in double precision
      const double pt64 = prob_f64(zt, st, ep), pd64 = prob_f64(zd, sd, ep);
      const double ratio = pd64 > 0.0 ? pt64 / pd64 : INFINITY;
      accept = static_cast<double>(u) < ratio;
      tie = fabs(static_cast<double>(u) - ratio) < DSPARK_TIE_EPS || !(pd64 > 0.0);
    }
  }
  const unsigned rej = __ballot_sync(0xFFFFFFFFu, has && !accept);
  const int m = rej ? __ffs(rej) - 1 : ell;
  const unsigned n_ties = __popc(__ballot_sync(0xFFFFFFFFu, tie && k <= m + 1));
  if (write_out && lane == 0 && n_ties) atomicAdd(ties, n_ties);

  if (write_out && pr && lane < gamma) {
    pr[2 * lane] = has ? pt : -1.f;
    pr[2 * lane + 1] = has ? pd : -1.f;
  }
  if (write_out) {
    if (lane < m)
      em[lane] = x;
    else if (lane > m && lane <= gamma)
      em[lane] = -1;
    if (lane == 0 && gamma == 32 && m < 32) em[32] = -1;
  }

  // descriptor of the token to sample after the block
  const int src = m < ell ? m : 0;
  const double Dm = __shfl_sync(0xFFFFFFFFu, Dk, src);
  const int Kt = __shfl_sync(0xFFFFFFFFu, st.K, src);
  if (lane == 0) {
    if (write_out) accepted_len[r] = m;
    ResampleDesc d;
    d.u = in.u_draw;
    if (!(d.u >= 0.f && d.u < 1.f)) {
      set_status(status, DSPARK_ERR_BAD_DATA);
      d.u = 0.f;
    }
    d.m = m;
    for (int i = 0; i < 2; ++i) d.pad[i] = 0;
    d.S_hi = d.S_lo = 0.f;
    d.E_hi = d.E_lo = 0.f;
    if (m < ell) {
      d.mode = kModeResidual;
      d.t_row = ws.row_list[start + m] >> 1;
      d.d_row = ws.row_list[start + ell + 1 + m] >> 1;
      d.K_t = Kt;
      const double D = Dm;
      d.D_hi = static_cast<float>(D);
      d.D_lo = static_cast<float>(D - static_cast<double>(d.D_hi));
      const double E = D - static_cast<double>(Kt);
      d.E_hi = static_cast<float>(E);
      d.E_lo = static_cast<float>(E - static_cast<double>(d.E_hi));
    } else {
      const RowStat sb = sh_rs[ell];  // the bonus row (position ell + 1)
      if (!sb.ok) set_status(status, DSPARK_ERR_BAD_DATA);
      d.mode = kModeTarget;
      d.t_row = ws.row_list[start + ell] >> 1;
      d.d_row = 0;
      d.K_t = sb.K == INT_MIN ? 0 : sb.K;
      d.D_hi = d.D_lo = 0.f;
    }
    *d_out = d;
  }
}

// ---------------------------------------------------------------------------
// k_resample: inverse-CDF draw from the residual or the target distribution
// ---------------------------------------------------------------------------
// Weight of token v, up to a factor common to the whole row:
//   target mode:   e_t(v) = 2^(z_t*c - K_t)                   (proportional to p_t)
//   residual mode: (e_t(v) - e_d(v))^+, e_d(v) = 2^(z_d*c + E) (proportional to
//                  max(0, p_t - p_d)), with E = D - K_t.
// p_d/p_t = 2^(-d2), d2 = (z_t - z_d)*c - D. For a token carrying much mass
// (e_t > 2^-8) with p_d close to p_t (0 < d2 < 1) the difference may cancel;
// there the weight is e_t * (1 - 2^(-d2)), the factor from its Taylor series
// in y = d2 ln 2 (ten terms: truncation below 1e-9 relative for y < ln 2).
// For d2 >= 1 the difference loses at most a few 1e-7 of relative precision.
struct WeightParams {
  int mode;
  float nK;          // -K_t
  float D_hi, D_lo;  // residual mode
  float E_hi, E_lo;
};

__device__ __forceinline__ WeightParams weight_params(const ResampleDesc& d) {
  return WeightParams{d.mode, -static_cast<float>(d.K_t), d.D_hi, d.D_lo, d.E_hi, d.E_lo};
}

// 1 - exp(-y) for 0 <= y < ln 2: y * sum_{k>=1} (-y)^(k-1) / k!, Horner form
__device__ __forceinline__ float one_minus_exp_neg_small(float y) {
  float t = -1.f / 3628800.f;                 // (-1)^(10+1) / 10!
  t = fmaf(t, y, 1.f / 362880.f);             // 1/9!
  t = fmaf(t, y, -1.f / 40320.f);
  t = fmaf(t, y, 1.f / 5040.f);
  t = fmaf(t, y, -1.f / 720.f);
  t = fmaf(t, y, 1.f / 120.f);
  t = fmaf(t, y, -1.f / 24.f);
  t = fmaf(t, y, 1.f / 6.f);
  t = fmaf(t, y, -0.5f);
  t = fmaf(t, y, 1.f);
  return t * y;
}

__device__ __forceinline__ float resample_weight(float zt, float zd, const WeightParams& w,
                                                 const ExpParams& ep) {
  const float e = exp_term(zt, w.nK, ep);
  if (w.mode == kModeTarget) return e;
  const float ed = ex2_approx(fmaf(zd, ep.c_lo, fmaf(zd, ep.c_hi, w.E_hi)) + w.E_lo);
  if (w.mode == kModeMin) return fminf(e, ed);  // no cancellation: a minimum
  float r = fmaxf(e - ed, 0.f);
  if (e > 0.00390625f) {  // rare: a heavy token
    const float dz = zt - zd;
    const float d2 = fmaf(dz, ep.c_hi, -w.D_hi) + fmaf(dz, ep.c_lo, -w.D_lo);
    if (!(d2 > 0.f))
      r = 0.f;
    else if (d2 < 1.f)
      r = e * one_minus_exp_neg_small(d2 * 0.6931471805599453f);
  }
  return r;
}

// The logits of a 16-byte vector as floats (bf16 from their 32-bit words).
template <typename Tin>
__device__ __forceinline__ void unpack_vec(const uint4& q, float (&z)[16 / sizeof(Tin)]) {
  if constexpr (sizeof(Tin) == 2) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      z[2 * k] = bf16_lo(w[k]);
      z[2 * k + 1] = bf16_hi(w[k]);
    }
  } else {
    z[0] = __uint_as_float(q.x);
    z[1] = __uint_as_float(q.y);
    z[2] = __uint_as_float(q.z);
    z[3] = __uint_as_float(q.w);
  }
}

template <typename Tin, int MODE>
__device__ __forceinline__ bool vec_weight_sum(const uint4& qt, const uint4& qd,
                                               const WeightParams& w, const ExpParams& ep,
                                               float& sum) {
  constexpr int E = 16 / sizeof(Tin);
  float zt[E], zd[E];
  unpack_vec<Tin>(qt, zt);
  if constexpr (MODE != kModeTarget) unpack_vec<Tin>(qd, zd);
  // The exponents of a token's target and draft terms (or of two target
  // terms) go through one two-lane FMA chain: each lane rounds exactly as
  // fmaf does, so the terms are bitwise those of the scalar form
  // (exp_term: fma(z, c_lo, fma(z, c_hi, nK)); the draft side then adds E_lo).
  const float2 chi = make_float2(ep.c_hi, ep.c_hi), clo = make_float2(ep.c_lo, ep.c_lo);
  float s = 0.f, emax = 0.f;
  if constexpr (MODE == kModeTarget) {
    const float2 k2 = make_float2(w.nK, w.nK);
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const float2 z2 = make_float2(zt[i], zt[i + 1]);
      const float2 a = __ffma2_rn(z2, clo, __ffma2_rn(z2, chi, k2));
      s += ex2_approx(a.x);
      s += ex2_approx(a.y);
    }
  } else {
    const float2 k2 = make_float2(w.nK, w.E_hi);
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float2 z2 = make_float2(zt[i], zd[i]);
      const float2 a = __ffma2_rn(z2, clo, __ffma2_rn(z2, chi, k2));
      const float e = ex2_approx(a.x);
      const float edv = ex2_approx(a.y + w.E_lo);
      if constexpr (MODE == kModeResidual) {
        emax = fmaxf(emax, e);
        s += fmaxf(e - edv, 0.f);
      } else {
        s += fminf(e, edv);
      }
    }
  }
  sum = s;
  return !(emax > 0.00390625f);
}

// The per-token sum of a vector holding a heavy token (rare).
template <typename Tin>
__device__ __forceinline__ float heavy_vec_sum(const uint4& qt, const uint4& qd,
                                               const WeightParams& wp, const ExpParams& ep) {
  constexpr int E = 16 / sizeof(Tin);
  const Tin* et = reinterpret_cast<const Tin*>(&qt);
  const Tin* ed = reinterpret_cast<const Tin*>(&qd);
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i)
    sum += resample_weight(to_float<Tin>(et[i]), to_float<Tin>(ed[i]), wp, ep);
  return sum;
}

template <typename Tin, int MODE>
__device__ __forceinline__ void span_sum_vec(const Tin* __restrict__ zt,
                                             const Tin* __restrict__ zd, int a, int b,
                                             const WeightParams& wp, const ExpParams& ep,
                                             int lane, LaneAcc& acc) {
  constexpr int E = 16 / sizeof(Tin);
  constexpr int NB = 2;
  const uint4* vt = reinterpret_cast<const uint4*>(zt);
  const uint4* vd = reinterpret_cast<const uint4*>(zd);
  const int v_end = b / E;
  for (int v0 = a / E + lane; v0 < v_end; v0 += 32 * NB) {
    uint4 qt[NB], qd[NB];
#pragma unroll
    for (int q = 0; q < NB; ++q) {
      const int vi = v0 + 32 * q;
      qt[q] = vi < v_end ? __ldg(vt + vi) : make_uint4(0u, 0u, 0u, 0u);
      if constexpr (MODE != kModeTarget)
        qd[q] = vi < v_end ? __ldg(vd + vi) : make_uint4(0u, 0u, 0u, 0u);
      else
        qd[q] = qt[q];
    }
#pragma unroll
    for (int q = 0; q < NB; ++q) {
      if (v0 + 32 * q >= v_end) break;
      float sum;
      if (!vec_weight_sum<Tin, MODE>(qt[q], qd[q], wp, ep, sum))
        sum = heavy_vec_sum<Tin>(qt[q], qd[q], wp, ep);
      kahan_add(acc, sum);
    }
  }
}

template <typename Tin, bool VEC>
__device__ void segment_sum(const Tin* __restrict__ zt, const Tin* __restrict__ zd, int a, int b,
                            const WeightParams& wp, const ExpParams& ep, int lane, float& out_hi,
                            float& out_lo) {
  const int mode = wp.mode;
  LaneAcc acc;
  if constexpr (VEC) {
    if (mode == kModeResidual)
      span_sum_vec<Tin, kModeResidual>(zt, zd, a, b, wp, ep, lane, acc);
    else if (mode == kModeMin)
      span_sum_vec<Tin, kModeMin>(zt, zd, a, b, wp, ep, lane, acc);
    else
      span_sum_vec<Tin, kModeTarget>(zt, zd, a, b, wp, ep, lane, acc);
  } else {
    for (int i = a + lane; i < b; i += 32) {
      const float z1 = to_float<Tin>(zt[i]);
      const float z2 = mode != kModeTarget ? to_float<Tin>(zd[i]) : z1;
      kahan_add(acc, resample_weight(z1, z2, wp, ep));
    }
  }
  float hi = acc.s, lo = -acc.comp;
  warp_two_sum(hi, lo);
  out_hi = hi;
  out_lo = lo;
}

// One warp scans the segment sums of a request: Z = their total, j = the
// first segment whose running sum exceeds u*Z (a segment with positive sum),
// P = the running sum before it; j = -1 if there is none. The sums may come
// from other CTAs of the running grid: they are read through L2.
__device__ void scan_segments(const ff* seg, int n_seg, float u, int lane, ff& Z_out, ff& P_out,
                              int& j_out) {
  constexpr int kHeld = 4;  // chunks of 32 sums kept in registers between the two passes
  const ff zero{0.f, 0.f};
  auto load = [&](int c) {
    return (c + lane < n_seg) ? ff{__ldcg(&seg[c + lane].hi), __ldcg(&seg[c + lane].lo)} : zero;
  };
  ff held[kHeld];
#pragma unroll
  for (int h = 0; h < kHeld; ++h) held[h] = load(32 * h);  // loads in flight together
  auto chunk = [&](int c) { return c < 32 * kHeld ? held[c >> 5] : load(c); };
  ff run = zero;
  for (int c = 0; c < n_seg; c += 32) {
    ff v = chunk(c);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const ff w = shfl_up_ff(v, o);
      if (lane >= o) v = ff_add(w, v);
    }
    run = ff_add(run, shfl_ff(v, 31));
  }
  const ff Z = run;
  const ff U = ff_mul(Z, ff{u, 0.f});
  int j = -1;
  ff P = zero;
  run = zero;
  for (int c = 0; c < n_seg && j < 0; c += 32) {
    ff v = chunk(c);
    const bool own_pos = v.hi > 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const ff w = shfl_up_ff(v, o);
      if (lane >= o) v = ff_add(w, v);
    }
    const ff incl = ff_add(run, v);
    const ff prev_incl = shfl_up_ff(incl, 1);
    const ff excl = lane == 0 ? run : prev_incl;  // running sum before this segment
    const unsigned hit =
        __ballot_sync(0xFFFFFFFFu, c + lane < n_seg && own_pos && ff_cmp(incl, U) > 0);
    if (hit) {
      const int l = __ffs(hit) - 1;
      j = c + l;
      P = shfl_ff(excl, l);
    }
    run = ff_add(run, shfl_ff(v, 31));
  }
  Z_out = Z;
  P_out = P;
  j_out = j;
}

// The whole CTA (256 threads) draws request r's token: finds the segment
// holding u*Z from the segment sums, then the token inside it. Running sums
// are float pairs (about 48 bits), far finer than the 1e-6*Z near-tie window.
template <typename Tin, bool VEC>
__device__ __noinline__ void pick_token(const Tin* __restrict__ tl, const Tin* __restrict__ dl, int V,
                           int n_seg, int gamma, const ExpParams& ep, const VerifyWs& ws,
                           const ResampleDesc& d, int r, int32_t* __restrict__ emitted,
                           uint32_t* ties, int32_t* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const Tin* zt = tl + d.t_row * static_cast<long long>(V);
  const Tin* zd = d.mode == kModeResidual ? dl + d.d_row * static_cast<long long>(V) : zt;
  WeightParams wp = weight_params(d);
  ff* seg = ws.seg_sum + static_cast<long long>(r) * n_seg;

  __shared__ ff sh_P, sh_Z;
  __shared__ int sh_j;
  __shared__ ff warp_tot[8];
  __shared__ unsigned long long sh_pick;  // (index << 1) | near-tie flag, min over threads
  __shared__ int sh_last_pos;
  int mode = d.mode;
  uint32_t flagged = 0;
  const ff zero{0.f, 0.f};
  for (int attempt = 0; attempt < 2; ++attempt) {
    if (warp == 0) {
      ff Z, P;
      int j;
      scan_segments(seg, n_seg, d.u, lane, Z, P, j);
      if (lane == 0) {
        sh_Z = Z;
        sh_P = P;
        sh_j = j;
      }
    }
    __syncthreads();
    if (sh_Z.hi > 0.f || attempt == 1) break;
    // zero residual mass (only in floating point): sample the target row instead
    mode = kModeTarget;
    wp.mode = kModeTarget;
    flagged = 1;
    for (int s2 = warp; s2 < n_seg; s2 += 8) {
      float hi, lo;
      segment_sum<Tin, VEC>(zt, zt, s2 * kSeg, min(V, (s2 + 1) * kSeg), wp, ep, lane, hi, lo);
      if (lane == 0) seg[s2] = ff_norm(hi, lo);
    }
    __syncthreads();
  }
  const ff Z = sh_Z, P = sh_P;
  const int j = sh_j;
  if (!(Z.hi > 0.f) || j < 0) {  // no mass at all: non-finite or empty rows
    if (tid == 0) {
      set_status(status, DSPARK_ERR_BAD_DATA);
      emitted[static_cast<long long>(r) * (gamma + 1) + d.m] = 0;
    }
    return;
  }
  const ff U = ff_mul(Z, ff{d.u, 0.f});
  const float win = static_cast<float>(DSPARK_TIE_EPS) * Z.hi;  // near-tie window
  // fine scan of segment j: 8 consecutive tokens per thread
  const int a = j * kSeg, b = min(V, a + kSeg);
  const int i0 = a + tid * 8;
  float w[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = i0 + q;
    w[q] = 0.f;
    if (i < b) {
      const float z1 = to_float<Tin>(zt[i]);
      const float z2 = mode == kModeResidual ? to_float<Tin>(zd[i]) : z1;
      w[q] = resample_weight(z1, z2, wp, ep);
    }
  }
  ff mine = zero;
#pragma unroll
  for (int q = 0; q < 8; ++q) mine = ff_add(mine, ff{w[q], 0.f});
  ff incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff t = shfl_up_ff(incl, o);
    if (lane >= o) incl = ff_add(t, incl);
  }
  ff ex = shfl_up_ff(incl, 1);
  if (lane == 0) ex = zero;
  if (tid == 0) {
    sh_pick = ~0ull;
    sh_last_pos = -1;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  ff before = ff_add(P, ex);
  for (int q = 0; q < warp; ++q) before = ff_add(before, warp_tot[q]);
  int last_pos = -1;
  for (int q = 0; q < 8; ++q)
    if (w[q] > 0.f) last_pos = i0 + q;
  // only the thread whose range can hold the cut walks its tokens
  if (ff_cmp(before, U) <= 0 && ff_cmp(ff_add(before, mine), U) > 0) {
    ff C = before;
    for (int q = 0; q < 8; ++q) {
      const ff below = C;
      C = ff_add(C, ff{w[q], 0.f});
      if (ff_cmp(C, U) > 0) {
        const bool near = ff_sub(U, below).hi < win || ff_sub(C, U).hi < win;
        atomicMin(&sh_pick, (static_cast<unsigned long long>(i0 + q) << 1) | (near ? 1ull : 0ull));
        break;
      }
    }
  }
  if (ff_cmp(before, U) <= 0 && last_pos >= 0) atomicMax(&sh_last_pos, last_pos);
  __syncthreads();
  if (tid == 0) {
    int y;
    if (sh_pick != ~0ull) {
      y = static_cast<int>(sh_pick >> 1);
      flagged |= static_cast<uint32_t>(sh_pick & 1ull);
    } else {  // rounding left u*Z beyond this segment's running sums
      y = sh_last_pos >= 0 ? sh_last_pos : a;
      flagged = 1;
    }
    emitted[static_cast<long long>(r) * (gamma + 1) + d.m] = y;
    if (flagged) atomicAdd(ties, 1u);
  }
}

// ---------------------------------------------------------------------------
// k_decide: ratio tests, residual / bonus segment sums and the draw, fused
// ---------------------------------------------------------------------------
constexpr int kDecideWarps = 8;
constexpr int kDecideMaxParts = 16;

// `parts` CTAs per request. Each one merges the request's row statistics
// and runs the ratio tests (cheap, so every part recomputes them and no part
// waits for another); part 0 writes the verification outputs. Each part sums
// the residual (or bonus) weights of its share of the 2048-token segments;
// the part that finishes last (ticket reset by k_plan) draws the token.
template <typename Tin, bool VEC>
__global__ void __launch_bounds__(kDecideWarps * 32, 6) k_decide(
    const Tin* __restrict__ tl, const Tin* __restrict__ dl, const int32_t* __restrict__ tokens,
    const float* __restrict__ uniforms, int B, int gamma, int V, int n_units, int n_seg,
    int parts, ExpParams ep, VerifyWs ws, int32_t* __restrict__ accepted_len,
    int32_t* __restrict__ emitted, float* __restrict__ probs_out, uint32_t* ties,
    int32_t* status) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  __shared__ RowStat sh_rs[2 * DSPARK_MAX_GAMMA + 1];
  __shared__ ResampleDesc sh_d;
  __shared__ int sh_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x / parts, part = blockIdx.x - r * parts;
  const bool lead = part == 0;
  const int start = ws.req_row_start[r], end = ws.req_row_start[r + 1];
  if (end == start) {  // invalid request (reported by k_plan): defined, in-bounds outputs
    if (lead && warp == 0) {
      int32_t* em = emitted + static_cast<long long>(r) * (gamma + 1);
      for (int k = lane; k <= gamma; k += 32) em[k] = -1;
      if (probs_out) {
        float* pr = probs_out + static_cast<long long>(r) * gamma * 2;
        for (int k = lane; k < gamma; k += 32) pr[2 * k] = pr[2 * k + 1] = -1.f;
      }
      if (lane == 0) accepted_len[r] = 0;
    }
    return;
  }
  // 0. the tested positions' inputs, in flight during the merge
  RatioIn rin{};
  if (warp == 0)
    rin = load_ratio_inputs<Tin>(tl, dl, tokens, uniforms, r, gamma, V, start,
                                 (end - start - 1) / 2, ws, lane);
  // 1. the request's row statistics (its rows' unit records are contiguous)
  merge_rows_block(ws.tiles + static_cast<long long>(start) * n_units, end - start, n_units,
                   sh_rs);
  __syncthreads();
  // 2. ratio tests and the first rejection
  if (warp == 0)
    ratio_tests<Tin>(rin, r, gamma, start, sh_rs, ep, ws, lead, accepted_len, emitted, probs_out,
                     ties, status, &sh_d, lane, end);
  __syncthreads();
  const ResampleDesc d = sh_d;
  // 3. this part's segment sums of the draw's weights
  const Tin* zt = tl + d.t_row * static_cast<long long>(V);
  const Tin* zd = d.mode == kModeResidual ? dl + d.d_row * static_cast<long long>(V) : zt;
  const WeightParams wp = weight_params(d);
  for (int sg = part * kDecideWarps + warp; sg < n_seg; sg += parts * kDecideWarps) {
    float hi, lo;
    segment_sum<Tin, VEC>(zt, zd, sg * kSeg, min(V, (sg + 1) * kSeg), wp, ep, lane, hi, lo);
    if (lane == 0) {
      ws.seg_sum[static_cast<long long>(r) * n_seg + sg] = ff_norm(hi, lo);
      __threadfence();  // before the part's ticket below
    }
  }
  // 4. the last part to finish draws the token
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    sh_last = atomicAdd(&ws.tickets[r], 1u) == static_cast<unsigned>(parts) - 1u;
  }
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  pick_token<Tin, VEC>(tl, dl, V, n_seg, gamma, ep, ws, d, r, emitted, ties, status);
}

// ---------------------------------------------------------------------------
// The decision pass for 16-byte aligned rows: k_desc, then k_resid
// ---------------------------------------------------------------------------
// k_desc: one CTA per request. It merges the request's rows, runs the ratio
// tests, writes accepted lengths, tokens and probabilities, and the
// descriptor of the token to draw after the block (mode kModeNone for an
// invalid request: nothing to draw).
template <typename Tin>
__global__ void __launch_bounds__(kDecideWarps * 32) k_desc(
    const Tin* __restrict__ tl, const Tin* __restrict__ dl, const int32_t* __restrict__ tokens,
    const float* __restrict__ uniforms, int gamma, int V, int n_units, ExpParams ep, VerifyWs ws,
    int32_t* __restrict__ accepted_len, int32_t* __restrict__ emitted,
    float* __restrict__ probs_out, uint32_t* ties, int32_t* status) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  __shared__ RowStat sh_rs[2 * DSPARK_MAX_GAMMA + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x;
  const int start = ws.req_row_start[r], end = ws.req_row_start[r + 1];
  if (end == start) {  // invalid request (reported by k_plan): defined, in-bounds outputs
    if (warp == 0) {
      int32_t* em = emitted + static_cast<long long>(r) * (gamma + 1);
      for (int k = lane; k <= gamma; k += 32) em[k] = -1;
      if (probs_out) {
        float* pr = probs_out + static_cast<long long>(r) * gamma * 2;
        for (int k = lane; k < gamma; k += 32) pr[2 * k] = pr[2 * k + 1] = -1.f;
      }
      if (lane == 0) {
        accepted_len[r] = 0;
        ws.desc[r].mode = kModeNone;
      }
    }
    return;
  }
  RatioIn rin{};
  if (warp == 0)
    rin = load_ratio_inputs<Tin>(tl, dl, tokens, uniforms, r, gamma, V, start,
                                 (end - start - 1) / 2, ws, lane);
  merge_rows_block(ws.tiles + static_cast<long long>(start) * n_units, end - start, n_units,
                   sh_rs);
  __syncthreads();
  if (warp == 0)
    ratio_tests<Tin>(rin, r, gamma, start, sh_rs, ep, ws, true, accepted_len, emitted, probs_out,
                     ties, status, ws.desc + r, lane, end);
}

// k_resid: per 2048-token segment, the weight sums of a list of jobs (one
// row pair each): for dspark_verify the residual (or bonus) weights of every
// request's draw, for dspark_acceptance the minima of every verified position.
// Persistent, W warps per CTA and one CTA per SM, like the streaming pass:
// warp w takes items w, w + GW, ... (item = s * n_jobs + j for segment s of
// job j: a warp's items fall in different segments, so that the segments rich
// in heavy tokens do not all land on the same warps) for all but the last
// 1/kDynamicDiv of them, which warps claim one at a time from a counter;
// items go through the warp's own ring of stages, each holding kRowPart bytes
// of the target row and kRowPart bytes of the draft row (only the target row
// for a bonus draw), fed by bulk copies; the ring runs on across items. The
// descriptors of a warp's next 32 fixed items are loaded together, one per
// lane, so that setting up an item costs shuffles, not a dependent load.
// k_pick then draws each request's token from the segment sums.
struct __align__(16) StageInfo {  // what a ring stage holds; written by lane 0
  float nK, E_hi, E_lo, D_hi, D_lo;
  int32_t mode;    // kModeResidual, kModeTarget or kModeMin
  int32_t bytes;   // bytes of each row in the stage
  int32_t out;     // the item's last stage: index of its sum; otherwise -1
};
static_assert(sizeof(StageInfo) == 32, "StageInfo layout");

// One lane's share of a batch of 32 items: the descriptor of item base + lane.
struct ItemRegs {
  const char* p_t;  // target-row segment
  const char* p_d;  // draft-row segment
  float nK, E_hi, E_lo, D_hi, D_lo;
  int32_t mode;     // kModeNone: nothing to sum
  int32_t bytes;    // bytes of each row in the segment
  int32_t out;      // index of the segment's sum
};

// Shared memory of the residual streamer: per warp STAGES stages of
// 2 * kRowPart bytes, then per warp STAGES barriers, then per warp STAGES
// stage records.
template <int W, int STAGES, int kRowPart>
__device__ __forceinline__ uint64_t* resid_bars(unsigned char* smem, int warp) {
  return reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(W) * STAGES * 2 * kRowPart) +
         warp * STAGES;
}

// The residual-sum streaming of one warp over its items (the body of k_resid):
// its ring barriers are initialised and the jobs visible. Returns early (with
// DSPARK_ERR_TIMEOUT recorded) if a copy never lands.
template <typename Tin, int W, int STAGES, int kRowPart>
__device__ __forceinline__ void resid_stream(const Tin* __restrict__ tl,
                                             const Tin* __restrict__ dl, int n_jobs, int V,
                                             int n_seg, const ExpParams& ep,
                                             const ResampleDesc* __restrict__ jobs,
                                             ff* __restrict__ sums, unsigned long long* claim,
                                             int32_t* status, unsigned char* smem) {
  constexpr int RPL = kRowPart / 16 / 32;  // 16-byte vectors per lane and row part
  constexpr int kSegBytes = kSeg * static_cast<int>(sizeof(Tin));
  constexpr int kStage = 2 * kRowPart;  // target part, then draft part
  constexpr unsigned kFull = 0xFFFFFFFFu;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* buf = smem + static_cast<size_t>(warp) * STAGES * kStage;
  uint64_t* bars = resid_bars<W, STAGES, kRowPart>(smem, warp);
  StageInfo* info =
      reinterpret_cast<StageInfo*>(smem + static_cast<size_t>(W) * STAGES * (kStage + 8)) +
      warp * STAGES;
  if (lane == 0) fence_proxy_async();  // the stages may have been written by generic stores

  const long long row_bytes = static_cast<long long>(V) * sizeof(Tin);
  const long long N = static_cast<long long>(n_jobs) * n_seg;
  const long long GW = static_cast<long long>(gridDim.x) * W;
  const long long g0 = static_cast<long long>(blockIdx.x) * W + warp;
  // items in fixed rounds for all but about 1/kDynamicDiv of them (warp g0:
  // items g0 + k GW, k < n_fixed), then claimed one at a time from *claim, so
  // that warps of CTAs that start late or run slow take fewer of the last ones
  const long long S = N - N / kDynamicDiv;  // items in fixed rounds
  const int n_fixed = g0 < S ? static_cast<int>((S - 1 - g0) / GW + 1) : 0;
  const long long dyn0 = S;

  auto describe = [&](long long i, ItemRegs& o) {  // the descriptor of item i
    o.mode = kModeNone;
    const int sg = static_cast<int>(i / n_jobs);
    const int j = static_cast<int>(i - static_cast<long long>(sg) * n_jobs);
    const ResampleDesc d = jobs[j];  // written by the previous kernel
    if (d.mode == kModeResidual || d.mode == kModeTarget || d.mode == kModeMin) {
      const long long off = static_cast<long long>(sg) * kSegBytes;
      const long long left = row_bytes - off;
      o.bytes = static_cast<int>(left < kSegBytes ? left : kSegBytes);
      o.p_t = reinterpret_cast<const char*>(tl) + d.t_row * row_bytes + off;
      o.p_d = reinterpret_cast<const char*>(dl) + d.d_row * row_bytes + off;
      o.nK = -static_cast<float>(d.K_t);
      o.E_hi = d.E_hi;
      o.E_lo = d.E_lo;
      o.D_hi = d.D_hi;
      o.D_lo = d.D_lo;
      o.out = j * n_seg + sg;
      o.mode = d.mode;
    }
  };
  ItemRegs mine{};
  auto load_batch = [&](int base) {  // lane l: the descriptor of fixed item base + l
    mine.mode = kModeNone;
    const int k = base + lane;
    if (k < n_fixed) describe(g0 + static_cast<long long>(k) * GW, mine);
  };

  // producer (warp-uniform state; lane 0 issues): item kp, its next stage pc
  int kp = 0, pc = 0, batch = -1;
  ItemRegs cur{};
  bool have = false;
  auto next_item = [&]() {  // sets up the next item with something to sum, if any
    have = false;
    for (; kp < n_fixed; ++kp) {
      if ((kp >> 5) != batch) {
        batch = kp >> 5;
        load_batch(batch << 5);
      }
      const int l = kp & 31;
      const int mode = __shfl_sync(kFull, mine.mode, l);
      if (mode == kModeNone) continue;
      cur.mode = mode;
      cur.p_t = reinterpret_cast<const char*>(
          __shfl_sync(kFull, reinterpret_cast<unsigned long long>(mine.p_t), l));
      cur.p_d = reinterpret_cast<const char*>(
          __shfl_sync(kFull, reinterpret_cast<unsigned long long>(mine.p_d), l));
      cur.nK = __shfl_sync(kFull, mine.nK, l);
      cur.E_hi = __shfl_sync(kFull, mine.E_hi, l);
      cur.E_lo = __shfl_sync(kFull, mine.E_lo, l);
      cur.D_hi = __shfl_sync(kFull, mine.D_hi, l);
      cur.D_lo = __shfl_sync(kFull, mine.D_lo, l);
      cur.bytes = __shfl_sync(kFull, mine.bytes, l);
      cur.out = __shfl_sync(kFull, mine.out, l);
      pc = 0;
      have = true;
      return;
    }
    for (;;) {  // the claimed items
      unsigned long long c = 0;
      if (lane == 0) c = atomicAdd(claim, 1ull);
      c = __shfl_sync(kFull, c, 0);
      const long long i = dyn0 + static_cast<long long>(c);
      if (i >= N) return;
      describe(i, cur);  // every lane the same item
      if (cur.mode == kModeNone) continue;
      pc = 0;
      have = true;
      return;
    }
  };
  auto issue = [&](int st) {  // one stage of the current item
    const int left = cur.bytes - pc * kRowPart;
    const uint32_t bytes = static_cast<uint32_t>(left < kRowPart ? left : kRowPart);
    const bool last = left <= kRowPart;
    if (lane == 0) {
      StageInfo in;
      in.nK = cur.nK;
      in.E_hi = cur.E_hi;
      in.E_lo = cur.E_lo;
      in.D_hi = cur.D_hi;
      in.D_lo = cur.D_lo;
      in.mode = cur.mode;
      in.bytes = static_cast<int>(bytes);
      in.out = last ? cur.out : -1;
      info[st] = in;
      const bool two = cur.mode != kModeTarget;
      mbar_arrive_expect_tx(&bars[st], two ? 2 * bytes : bytes);
      bulk_g2s(buf + st * kStage, cur.p_t + static_cast<long long>(pc) * kRowPart, bytes,
               &bars[st]);
      if (two)
        bulk_g2s(buf + st * kStage + kRowPart, cur.p_d + static_cast<long long>(pc) * kRowPart,
                 bytes, &bars[st]);
    }
    ++pc;
    if (last) {
      ++kp;
      next_item();
    }
  };

  int inflight = 0;
  next_item();
  while (inflight < STAGES && have) issue(inflight++);

  int stage = 0;
  uint32_t phase = 0;
  LaneAcc acc;
  while (inflight > 0) {
    // every lane waits (each gets the barrier's acquire); the give-up decision is warp-uniform
    if (!__all_sync(kFull, mbar_wait(&bars[stage], phase))) {
      if (lane == 0) set_status(status, DSPARK_ERR_TIMEOUT);
      for (int q = 0; q < inflight; ++q) {  // let the copies in flight land before leaving
        int s2 = stage + q;
        uint32_t p2 = phase;
        if (s2 >= STAGES) {
          s2 -= STAGES;
          p2 ^= 1u;
        }
        (void)mbar_wait(&bars[s2], p2);
      }
      return;
    }
    const StageInfo in = info[stage];
    const bool two = in.mode != kModeTarget;
    uint4 v[2 * RPL];
    const uint4* sp = reinterpret_cast<const uint4*>(buf + stage * kStage);
    const int n_vec = in.bytes == kRowPart ? RPL : (in.bytes / 16 - lane + 31) / 32;
#pragma unroll
    for (int q = 0; q < RPL; ++q) {
      const int idx = q * 32 + lane;
      const bool ok = q < n_vec;
      v[q] = ok ? sp[idx] : make_uint4(0u, 0u, 0u, 0u);
      v[RPL + q] = (ok && two) ? sp[kRowPart / 16 + idx] : v[q];
    }
    __syncwarp();
    const int freed = stage;
    if (++stage == STAGES) {
      stage = 0;
      phase ^= 1u;
    }
    --inflight;
    if (have) {  // the ring was full: the freed stage is the next one to fill
      if (lane == 0) fence_proxy_async();
      issue(freed);
      ++inflight;
    }

    const WeightParams wp{in.mode, in.nK, in.D_hi, in.D_lo, in.E_hi, in.E_lo};
#pragma unroll
    for (int q = 0; q < RPL; ++q) {
      if (q >= n_vec) break;
      float sum;
      bool light = true;
      if (in.mode == kModeResidual)
        light = vec_weight_sum<Tin, kModeResidual>(v[q], v[RPL + q], wp, ep, sum);
      else if (in.mode == kModeMin)
        (void)vec_weight_sum<Tin, kModeMin>(v[q], v[RPL + q], wp, ep, sum);
      else
        (void)vec_weight_sum<Tin, kModeTarget>(v[q], v[q], wp, ep, sum);
      if (!light) sum = heavy_vec_sum<Tin>(v[q], v[RPL + q], wp, ep);
      kahan_add(acc, sum);
    }
    if (in.out >= 0) {
      float hi = acc.s, lo = -acc.comp;
      warp_two_sum(hi, lo);
      acc = LaneAcc();
      if (lane == 0) sums[in.out] = ff_norm(hi, lo);
    }
  }
}

template <typename Tin, int W, int STAGES, int kRowPart>
__global__ void __launch_bounds__(W * 32, 1)
    k_resid(const Tin* __restrict__ tl, const Tin* __restrict__ dl, int n_jobs, int V, int n_seg,
            ExpParams ep, const ResampleDesc* __restrict__ jobs, ff* __restrict__ sums,
            unsigned long long* claim, int32_t* status) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    uint64_t* bars = resid_bars<W, STAGES, kRowPart>(smem, warp);
    for (int st = 0; st < STAGES; ++st) mbar_init(&bars[st], 1);
    fence_barrier_init();
  }
  __syncwarp();
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  resid_stream<Tin, W, STAGES, kRowPart>(tl, dl, n_jobs, V, n_seg, ep, jobs, sums, claim, status,
                                          smem);
}

// k_pick: one CTA per request draws the token after the block from the
// segment sums k_resid wrote (nothing to do for an invalid request).
template <typename Tin>
__global__ void __launch_bounds__(kDecideWarps * 32)
    k_pick(const Tin* __restrict__ tl, const Tin* __restrict__ dl, int gamma, int V, int n_seg,
           ExpParams ep, VerifyWs ws, int32_t* __restrict__ emitted, uint32_t* ties,
           int32_t* status) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  const int r = blockIdx.x;
  const ResampleDesc d = ws.desc[r];
  if (d.mode != kModeResidual && d.mode != kModeTarget) return;
  pick_token<Tin, true>(tl, dl, V, n_seg, gamma, ep, ws, d, r, emitted, ties, status);
}

// ---------------------------------------------------------------------------
// dspark_acceptance: sum_v min(p_t^k, p_d^k) for every verified position
// ---------------------------------------------------------------------------
// k_rate_desc: one CTA per request merges its rows and writes one job per
// position: the row pair, K_t, E = D - K_t and the target row's sum S_t, so that
// the rate is sum_v min(e_t(v), e_d(v)) / S_t with e_d = 2^(z_d*c + E).
// Positions beyond l_r (and every position of an invalid request) get no job.
__global__ void __launch_bounds__(kDecideWarps * 32)
    k_rate_desc(int gamma, int n_units, VerifyWs ws, ResampleDesc* __restrict__ jobs,
                int32_t* status) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  __shared__ RowStat sh_rs[2 * DSPARK_MAX_GAMMA + 1];
  const int r = blockIdx.x;
  const int start = ws.req_row_start[r], end = ws.req_row_start[r + 1];
  const int ell = end > start ? (end - start - 1) / 2 : 0;
  if (end > start)
    merge_rows_block(ws.tiles + static_cast<long long>(start) * n_units, end - start, n_units,
                     sh_rs);
  __syncthreads();
  for (int k = threadIdx.x; k < gamma; k += blockDim.x) {
    ResampleDesc d{};
    d.mode = kModeNone;
    if (k < ell) {
      const RowStat st = sh_rs[k], sd = sh_rs[ell + 1 + k];
      if (!st.ok || !sd.ok) {
        set_status(status, DSPARK_ERR_BAD_DATA);
      } else {
        const double D = static_cast<double>(st.K - sd.K) +
                         log2((static_cast<double>(st.S_hi) + st.S_lo) /
                              (static_cast<double>(sd.S_hi) + sd.S_lo));
        const double E = D - static_cast<double>(st.K);
        d.t_row = ws.row_list[start + k] >> 1;
        d.d_row = ws.row_list[start + ell + 1 + k] >> 1;
        d.K_t = st.K;
        d.E_hi = static_cast<float>(E);
        d.E_lo = static_cast<float>(E - static_cast<double>(d.E_hi));
        d.S_hi = st.S_hi;
        d.S_lo = st.S_lo;
        d.m = k;
        d.mode = kModeMin;
      }
    }
    jobs[static_cast<long long>(r) * gamma + k] = d;
  }
}

// The minima's segment sums for rows that are not 16-byte aligned: one warp per
// (job, segment), plain loads.
template <typename Tin>
__global__ void __launch_bounds__(256)
    k_rate_sum_plain(const Tin* __restrict__ tl, const Tin* __restrict__ dl, int n_jobs, int V,
                     int n_seg, ExpParams ep, const ResampleDesc* __restrict__ jobs,
                     ff* __restrict__ sums) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long n_items = static_cast<long long>(n_jobs) * n_seg;
  const long long GW = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long it = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       it < n_items; it += GW) {
    const int j = static_cast<int>(it / n_seg), sg = static_cast<int>(it - (it / n_seg) * n_seg);
    const ResampleDesc d = jobs[j];
    if (d.mode != kModeMin) continue;
    float hi, lo;
    segment_sum<Tin, false>(tl + d.t_row * static_cast<long long>(V),
                            dl + d.d_row * static_cast<long long>(V), sg * kSeg,
                            min(V, (sg + 1) * kSeg), weight_params(d), ep, lane, hi, lo);
    if (lane == 0) sums[it] = ff_norm(hi, lo);
  }
}

// k_rate_finish: one warp per position adds its segment sums (lanes take
// every 32nd sum, then a butterfly, all in float pairs) and divides by S_t;
// -1 where there is no job.
constexpr int kFinishWarps = 8;
__global__ void __launch_bounds__(kFinishWarps * 32)
    k_rate_finish(int n_jobs, int n_seg, const ResampleDesc* __restrict__ jobs,
                  const ff* __restrict__ sums, float* __restrict__ rates) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x * kFinishWarps + (threadIdx.x >> 5);
  if (j >= n_jobs) return;  // whole warps only
  const ResampleDesc d = jobs[j];
  if (d.mode != kModeMin) {
    if (lane == 0) rates[j] = -1.f;
    return;
  }
  const ff* s = sums + static_cast<long long>(j) * n_seg;
  ff t{0.f, 0.f};
  for (int sg = lane; sg < n_seg; sg += 32) t = ff_add(t, s[sg]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const ff u{__shfl_xor_sync(0xFFFFFFFFu, t.hi, o), __shfl_xor_sync(0xFFFFFFFFu, t.lo, o)};
    t = ff_add(t, u);
  }
  if (lane == 0) {
    const double rate =
        (static_cast<double>(t.hi) + t.lo) / (static_cast<double>(d.S_hi) + d.S_lo);
    rates[j] = static_cast<float>(rate);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
constexpr int kStreamWarps = 16;
constexpr int kStages = 3;

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int decide_ctas_per_sm = 1;  // resident k_decide CTAs per SM
};
std::mutex g_mutex;
DeviceState g_devices[128];

constexpr size_t tma_smem_bytes() {
  return static_cast<size_t>(kStreamWarps) * kStages *
         (kChunkBytes + sizeof(uint64_t) + sizeof(ChunkRec));
}
// k_resid: 16 warps per SM, each with a ring of 3 stages of 2 KB per row (32
// warps with 1 KB parts measured slower: the per-stage work halves, its
// overhead does not)
constexpr int kResidWarps = 16;
constexpr int kResidStages = 3;
constexpr int kResidPart = 2048;
constexpr size_t resid_smem_bytes() {
  return static_cast<size_t>(kResidWarps) * kResidStages *
         (2 * kResidPart + sizeof(uint64_t) + sizeof(StageInfo));
}
static_assert(resid_smem_bytes() <= 227 * 1024, "shared memory of k_resid");

int device_setup(int& sms, int& decide_per_sm) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return DSPARK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_devices[dev];
  if (!s.ready) {
    if (cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    if (cudaFuncSetAttribute(k_rowstats_tma<uint16_t, kStreamWarps, kStages>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tma_smem_bytes())) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    if (cudaFuncSetAttribute(k_rowstats_tma<float, kStreamWarps, kStages>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tma_smem_bytes())) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    if (cudaFuncSetAttribute(k_resid<uint16_t, kResidWarps, kResidStages, kResidPart>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(resid_smem_bytes())) != cudaSuccess ||
        cudaFuncSetAttribute(k_resid<float, kResidWarps, kResidStages, kResidPart>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(resid_smem_bytes())) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_decide<uint16_t, false>,
                                                      kDecideWarps * 32, 0) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    s.decide_ctas_per_sm = occ > 0 ? occ : 1;
    s.ready = true;
  }
  sms = s.sms;
  decide_per_sm = s.decide_ctas_per_sm;
  return DSPARK_OK;
}


ExpParams exp_params(float temperature) {
  ExpParams ep;
  ep.c_d = 1.4426950408889634 / static_cast<double>(temperature);  // log2(e) / T
  float hi = static_cast<float>(ep.c_d);
  if (static_cast<double>(hi) > ep.c_d) hi = std::nextafter(hi, 0.0f);
  ep.c_hi = hi;
  ep.c_lo = static_cast<float>(ep.c_d - static_cast<double>(hi));
  if (!(ep.c_lo > 0.0f)) ep.c_lo = 1e-30f;  // keeps c_lo * (-inf) = -inf
  return ep;
}

VerifyWs carve_verify_ws(void* base, int B, int gamma, int V) {
  char* p = static_cast<char*>(base);
  VerifyWs ws;
  ws.hdr = reinterpret_cast<WsHeader*>(p);
  p += 256;
  ws.req_row_start = reinterpret_cast<int32_t*>(p);
  p += DSPARK_ALIGN256((static_cast<size_t>(B) + 1) * 4);
  ws.row_list = reinterpret_cast<int64_t*>(p);
  p += DSPARK_ALIGN256(DSPARK_MAX_ROWS(B, gamma) * 8);
  ws.tiles = reinterpret_cast<TileStat*>(p);
  p += DSPARK_ALIGN256(DSPARK_MAX_ROWS(B, gamma) * DSPARK_TILES_PER_ROW(V) * 16);
  ws.desc = reinterpret_cast<ResampleDesc*>(p);
  p += DSPARK_ALIGN256(static_cast<size_t>(B) * 64);
  ws.seg_sum = reinterpret_cast<ff*>(p);
  p += DSPARK_ALIGN256(static_cast<size_t>(B) * DSPARK_SEGS_PER_ROW(V) * 8);
  ws.tickets = reinterpret_cast<uint32_t*>(p);
  return ws;
}

template <typename Tin>
int launch_verify(const Tin* tl, const Tin* dl, const int32_t* tokens, const int32_t* vlen,
                  const float* uni, float temperature, int B, int gamma, int V,
                  const int64_t* toff, const int64_t* doff, int32_t* acc, int32_t* emitted,
                  float* probs, uint32_t* ties, int32_t* status, void* workspace,
                  cudaStream_t stream, cudaEvent_t* ev) {
  int sms = 0, decide_per_sm = 1;
  if (int rc = device_setup(sms, decide_per_sm)) return rc;
  VerifyWs ws = carve_verify_ws(workspace, B, gamma, V);
  uint32_t* tie_ctr = ties ? ties : &ws.hdr->ties_scratch;
  const ExpParams ep = exp_params(temperature);
  const int unit_elems = kUnitBytes / static_cast<int>(sizeof(Tin));
  const int n_units = (V + unit_elems - 1) / unit_elems;
  const int n_seg = (V + kSeg - 1) / kSeg;

  if (ev && cudaEventRecord(ev[0], stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (launch_pdl(k_plan, 1, 1024, 0, stream, vlen, toff, doff, B, gamma, ws, tie_ctr, status) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (ev && cudaEventRecord(ev[1], stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (B == 0) {
    if (ev && (cudaEventRecord(ev[2], stream) != cudaSuccess ||
               cudaEventRecord(ev[3], stream) != cudaSuccess))
      return DSPARK_ERR_CUDA;
    return DSPARK_OK;
  }

  const bool aligned = (static_cast<size_t>(V) * sizeof(Tin)) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(tl) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(dl) % 16 == 0;
  const long long max_units = static_cast<long long>(DSPARK_MAX_ROWS(B, gamma)) * n_units;
  if (aligned) {
    const long long want = (max_units + kStreamWarps - 1) / kStreamWarps;
    const int grid = static_cast<int>(want < sms ? want : sms);
    if (launch_pdl(k_rowstats_tma<Tin, kStreamWarps, kStages>, grid, kStreamWarps * 32,
                   tma_smem_bytes(), stream, tl, dl, V, n_units, ws, ep, status) != cudaSuccess)
      return DSPARK_ERR_CUDA;
  } else {
    const long long want = (max_units + 7) / 8;
    const int grid = static_cast<int>(want < 4LL * sms ? want : 4LL * sms);
    if (launch_pdl(k_rowstats_plain<Tin>, grid, 256, 0, stream, tl, dl, V, n_units, ws, ep,
                   status) != cudaSuccess)
      return DSPARK_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  if (ev && cudaEventRecord(ev[2], stream) != cudaSuccess) return DSPARK_ERR_CUDA;

  if (aligned) {
    // decisions per request, then the residual segments by a persistent streamer
    if (launch_pdl(k_desc<Tin>, B, kDecideWarps * 32, 0, stream, tl, dl, tokens, uni, gamma, V,
                   n_units, ep, ws, acc, emitted, probs, tie_ctr, status) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    const long long items = static_cast<long long>(B) * n_seg;
    const long long want = (items + kResidWarps - 1) / kResidWarps;
    const int grid = static_cast<int>(want < sms ? want : sms);
    if (launch_pdl(k_resid<Tin, kResidWarps, kResidStages, kResidPart>, grid, kResidWarps * 32,
                   resid_smem_bytes(), stream, tl, dl, B, V, n_seg, ep,
                   static_cast<const ResampleDesc*>(ws.desc), ws.seg_sum, &ws.hdr->next_item,
                   status) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    if (launch_pdl(k_pick<Tin>, B, kDecideWarps * 32, 0, stream, tl, dl, gamma, V, n_seg, ep, ws,
                   emitted, tie_ctr, status) != cudaSuccess)
      return DSPARK_ERR_CUDA;
  } else {
    // CTAs per request: as many as one wave of resident CTAs holds (at least
    // one, and no more than there are segments to share)
    int parts = static_cast<int>(static_cast<long long>(decide_per_sm) * sms / B);
    parts = parts < 1 ? 1 : (parts > kDecideMaxParts ? kDecideMaxParts : parts);
    const int seg_groups = (n_seg + kDecideWarps - 1) / kDecideWarps;
    if (parts > seg_groups) parts = seg_groups;
    if (launch_pdl(k_decide<Tin, false>, dim3(static_cast<unsigned>(B) * parts),
                   kDecideWarps * 32, 0, stream, tl, dl, tokens, uni, B, gamma, V, n_units, n_seg,
                   parts, ep, ws, acc, emitted, probs, tie_ctr, status) != cudaSuccess)
      return DSPARK_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  if (ev && cudaEventRecord(ev[3], stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

}  // namespace dspark

namespace dspark {

int verify_entry(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                 const int32_t* verify_len, const float* uniforms, float temperature,
                 int32_t dtype, int32_t B, int32_t gamma, int32_t V,
                 const int64_t* target_row_off, const int64_t* draft_row_off,
                 int32_t* accepted_len, int32_t* emitted_tokens, float* probs_out,
                 uint32_t* near_tie_count, int32_t* device_status, void* workspace,
                 size_t workspace_bytes, cudaStream_t s, cudaEvent_t* ev) {
  // B times the CTAs per request indexes a grid dimension; V keeps segment offsets in int
  if (B < 0 || B > 65535 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || V < 1 || V > (1 << 30))
    return DSPARK_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return DSPARK_ERR_INVALID_ARG;
  if (dtype != DSPARK_F32 && dtype != DSPARK_BF16) return DSPARK_ERR_INVALID_ARG;
  if (!device_status) return DSPARK_ERR_INVALID_ARG;
  if ((target_row_off == nullptr) != (draft_row_off == nullptr)) return DSPARK_ERR_INVALID_ARG;
  if (B > 0 && (!target_logits || !draft_logits || !draft_tokens || !verify_len || !uniforms ||
                !accepted_len || !emitted_tokens))
    return DSPARK_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < DSPARK_VERIFY_WS_BYTES(B, gamma, V) ||
      reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return DSPARK_ERR_WORKSPACE;
  if (dtype == DSPARK_BF16)
    return launch_verify<uint16_t>(
        static_cast<const uint16_t*>(target_logits), static_cast<const uint16_t*>(draft_logits),
        draft_tokens, verify_len, uniforms, temperature, B, gamma, V, target_row_off,
        draft_row_off, accepted_len, emitted_tokens, probs_out, near_tie_count, device_status,
        workspace, s, ev);
  return launch_verify<float>(static_cast<const float*>(target_logits),
                              static_cast<const float*>(draft_logits), draft_tokens, verify_len,
                              uniforms, temperature, B, gamma, V, target_row_off, draft_row_off,
                              accepted_len, emitted_tokens, probs_out, near_tie_count,
                              device_status, workspace, s, ev);
}

}  // namespace dspark

extern "C" int dspark_verify(const void* target_logits, const void* draft_logits,
                             const int32_t* draft_tokens, const int32_t* verify_len,
                             const float* uniforms, float temperature, int32_t dtype, int32_t B,
                             int32_t gamma, int32_t V, const int64_t* target_row_off,
                             const int64_t* draft_row_off, int32_t* accepted_len,
                             int32_t* emitted_tokens, float* probs_out,
                             uint32_t* near_tie_count, int32_t* device_status, void* workspace,
                             size_t workspace_bytes, struct CUstream_st* stream) {
  return dspark::verify_entry(target_logits, draft_logits, draft_tokens, verify_len, uniforms,
                              temperature, dtype, B, gamma, V, target_row_off, draft_row_off,
                              accepted_len, emitted_tokens, probs_out, near_tie_count,
                              device_status, workspace, workspace_bytes,
                              reinterpret_cast<cudaStream_t>(stream), nullptr);
}

extern "C" int dspark_verify_timed(const void* target_logits, const void* draft_logits,
                                   const int32_t* draft_tokens, const int32_t* verify_len,
                                   const float* uniforms, float temperature, int32_t dtype,
                                   int32_t B, int32_t gamma, int32_t V,
                                   const int64_t* target_row_off, const int64_t* draft_row_off,
                                   int32_t* accepted_len, int32_t* emitted_tokens,
                                   float* probs_out, uint32_t* near_tie_count,
                                   int32_t* device_status, void* workspace,
                                   size_t workspace_bytes, struct CUstream_st* stream,
                                   struct CUevent_st** events) {
  if (!events) return DSPARK_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i)
    if (!events[i]) return DSPARK_ERR_INVALID_ARG;
  cudaEvent_t ev[4] = {events[0], events[1], events[2], events[3]};
  return dspark::verify_entry(target_logits, draft_logits, draft_tokens, verify_len, uniforms,
                              temperature, dtype, B, gamma, V, target_row_off, draft_row_off,
                              accepted_len, emitted_tokens, probs_out, near_tie_count,
                              device_status, workspace, workspace_bytes,
                              reinterpret_cast<cudaStream_t>(stream), ev);
}

// ---------------------------------------------------------------------------
// dspark_verify_static: the same verification with library-owned scratch, for
// callers that cannot allocate device memory (no counterpart in the paper).
// ---------------------------------------------------------------------------
namespace dspark {

// One array per device that loads the library, kept until the process exits
// and shared by every call on that device. Its contents need no clearing
// between calls: k_plan resets the tickets and counters each call relies on.
static __device__ __align__(256) unsigned char g_static_ws[DSPARK_STATIC_WS_BYTES];

std::mutex g_static_mutex;
struct StaticWsAddress {
  unsigned long long ctx_id;  // context the address belongs to (0: unknown)
  void* ptr;
};
StaticWsAddress g_static_ws_ptr[128];  // device address of g_static_ws, per device

// The unique ID of the calling thread's current context, or 0 when there is
// none or the driver cannot say. IDs are never reused within a process, so a
// context created after a device reset gets a new one even if it lands at the
// same address.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(fn);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// In host code g_static_ws names a host-side stand-in, not device memory. Its
// device address is looked up with the device current, once per device and
// context: a device reset (cudaDeviceReset, or another library resetting the
// primary context) reloads the module at a new address, and the context ID
// changes with it, so the lookup is repeated then. Without a context ID from
// the driver every call looks the address up.
int static_ws_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return DSPARK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  StaticWsAddress& c = g_static_ws_ptr[dev];
  const unsigned long long id = current_context_id();
  if (id == 0 || c.ctx_id != id || c.ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr)
      return DSPARK_ERR_CUDA;
    // the lookup makes the primary context current if none was
    c.ctx_id = id ? id : current_context_id();
    c.ptr = p;
  }
  *out = c.ptr;
  return DSPARK_OK;
}

}  // namespace dspark

extern "C" int dspark_verify_static(const void* target_logits, const void* draft_logits,
                                    const int32_t* draft_tokens, const int32_t* verify_len,
                                    const float* uniforms, float temperature, int32_t dtype,
                                    int32_t B, int32_t gamma, int32_t V,
                                    const int64_t* target_row_off, const int64_t* draft_row_off,
                                    int32_t* accepted_len, int32_t* emitted_tokens,
                                    float* probs_out, uint32_t* near_tie_count,
                                    int32_t* device_status, struct CUstream_st* stream) {
  using namespace dspark;
  if (B < 0 || B > 65535 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || V < 1 || V > (1 << 30))
    return DSPARK_ERR_INVALID_ARG;
  if (DSPARK_VERIFY_WS_BYTES(B, gamma, V) > DSPARK_STATIC_WS_BYTES) return DSPARK_ERR_TOO_LARGE;
  void* ws = nullptr;
  if (int rc = static_ws_address(&ws)) return rc;
  return dspark_verify(target_logits, draft_logits, draft_tokens, verify_len, uniforms,
                       temperature, dtype, B, gamma, V, target_row_off, draft_row_off,
                       accepted_len, emitted_tokens, probs_out, near_tie_count, device_status,
                       ws, DSPARK_STATIC_WS_BYTES, stream);
}

// ---------------------------------------------------------------------------
// dspark_acceptance (equation 8 per position; section 3.2.1's label)
// ---------------------------------------------------------------------------
namespace dspark {

// The acceptance probabilities of every verified position from the row
// statistics already in the workspace (k_plan and the streaming pass ran):
// k_rate_desc, the minima's segment sums, k_rate_finish. The jobs and their
// sums follow the verification workspace (DSPARK_ACCEPTANCE_WS_BYTES).
template <typename Tin>
int launch_rates(const Tin* tl, const Tin* dl, int B, int gamma, int V, float temperature,
                 float* rates, int32_t* status, void* workspace, cudaStream_t stream,
                 bool aligned) {
  int sms = 0, decide_per_sm = 1;
  if (int rc = device_setup(sms, decide_per_sm)) return rc;
  VerifyWs ws = carve_verify_ws(workspace, B, gamma, V);
  char* p = static_cast<char*>(workspace) + DSPARK_VERIFY_WS_BYTES(B, gamma, V);
  ResampleDesc* jobs = reinterpret_cast<ResampleDesc*>(p);
  p += DSPARK_ALIGN256(static_cast<size_t>(B) * gamma * 64);
  ff* sums = reinterpret_cast<ff*>(p);
  const ExpParams ep = exp_params(temperature);
  const int unit_elems = kUnitBytes / static_cast<int>(sizeof(Tin));
  const int n_units = (V + unit_elems - 1) / unit_elems;
  const int n_seg = (V + kSeg - 1) / kSeg;
  const int n_jobs = B * gamma;
  if (launch_pdl(k_rate_desc, B, kDecideWarps * 32, 0, stream, gamma, n_units, ws, jobs,
                 status) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  const long long items = static_cast<long long>(n_jobs) * n_seg;
  cudaError_t e;
  if (aligned) {
    const long long want = (items + kResidWarps - 1) / kResidWarps;
    e = launch_pdl(k_resid<Tin, kResidWarps, kResidStages, kResidPart>,
                   static_cast<int>(want < sms ? want : sms), kResidWarps * 32, resid_smem_bytes(),
                   stream, tl, dl, n_jobs, V, n_seg, ep, static_cast<const ResampleDesc*>(jobs),
                   sums, &ws.hdr->next_rate, status);
  } else {
    const long long want = (items + 7) / 8;
    e = launch_pdl(k_rate_sum_plain<Tin>, static_cast<int>(want < 4LL * sms ? want : 4LL * sms),
                   256, 0, stream, tl, dl, n_jobs, V, n_seg, ep,
                   static_cast<const ResampleDesc*>(jobs), sums);
  }
  if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  if (launch_pdl(k_rate_finish, (n_jobs + kFinishWarps - 1) / kFinishWarps, kFinishWarps * 32, 0,
                 stream, n_jobs, n_seg, static_cast<const ResampleDesc*>(jobs),
                 static_cast<const ff*>(sums), rates) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

template <typename Tin>
int launch_acceptance(const Tin* tl, const Tin* dl, const int32_t* vlen, float temperature,
                      int B, int gamma, int V, const int64_t* toff, const int64_t* doff,
                      float* rates, int32_t* status, void* workspace, cudaStream_t stream) {
  int sms = 0, decide_per_sm = 1;
  if (int rc = device_setup(sms, decide_per_sm)) return rc;
  VerifyWs ws = carve_verify_ws(workspace, B, gamma, V);
  const ExpParams ep = exp_params(temperature);
  const int unit_elems = kUnitBytes / static_cast<int>(sizeof(Tin));
  const int n_units = (V + unit_elems - 1) / unit_elems;
  if (launch_pdl(k_plan, 1, 1024, 0, stream, vlen, toff, doff, B, gamma, ws,
                 &ws.hdr->ties_scratch, status) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (B == 0) return DSPARK_OK;
  const bool aligned = (static_cast<size_t>(V) * sizeof(Tin)) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(tl) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(dl) % 16 == 0;
  const long long max_units = static_cast<long long>(DSPARK_MAX_ROWS(B, gamma)) * n_units;
  cudaError_t e;
  if (aligned) {
    const long long want = (max_units + kStreamWarps - 1) / kStreamWarps;
    e = launch_pdl(k_rowstats_tma<Tin, kStreamWarps, kStages>,
                   static_cast<int>(want < sms ? want : sms), kStreamWarps * 32, tma_smem_bytes(),
                   stream, tl, dl, V, n_units, ws, ep, status);
  } else {
    const long long want = (max_units + 7) / 8;
    e = launch_pdl(k_rowstats_plain<Tin>, static_cast<int>(want < 4LL * sms ? want : 4LL * sms),
                   256, 0, stream, tl, dl, V, n_units, ws, ep, status);
  }
  if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  return launch_rates<Tin>(tl, dl, B, gamma, V, temperature, rates, status, workspace, stream,
                           aligned);
}

}  // namespace dspark

extern "C" int dspark_acceptance(const void* target_logits, const void* draft_logits,
                                 const int32_t* verify_len, float temperature, int32_t dtype,
                                 int32_t B, int32_t gamma, int32_t V,
                                 const int64_t* target_row_off, const int64_t* draft_row_off,
                                 float* rates, int32_t* device_status, void* workspace,
                                 size_t workspace_bytes, struct CUstream_st* stream) {
  using namespace dspark;
  if (B < 0 || B > 65535 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || V < 1 || V > (1 << 30))
    return DSPARK_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return DSPARK_ERR_INVALID_ARG;
  if (dtype != DSPARK_F32 && dtype != DSPARK_BF16) return DSPARK_ERR_INVALID_ARG;
  if (!device_status) return DSPARK_ERR_INVALID_ARG;
  if ((target_row_off == nullptr) != (draft_row_off == nullptr)) return DSPARK_ERR_INVALID_ARG;
  if (B > 0 && (!target_logits || !draft_logits || !verify_len || !rates))
    return DSPARK_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < DSPARK_ACCEPTANCE_WS_BYTES(B, gamma, V) ||
      reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return DSPARK_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == DSPARK_BF16)
    return launch_acceptance<uint16_t>(static_cast<const uint16_t*>(target_logits),
                                       static_cast<const uint16_t*>(draft_logits), verify_len,
                                       temperature, B, gamma, V, target_row_off, draft_row_off,
                                       rates, device_status, workspace, s);
  return launch_acceptance<float>(static_cast<const float*>(target_logits),
                                  static_cast<const float*>(draft_logits), verify_len,
                                  temperature, B, gamma, V, target_row_off, draft_row_off, rates,
                                  device_status, workspace, s);
}

// ---------------------------------------------------------------------------
// dspark_verify_rates: dspark_verify, then the acceptance probabilities of
// every verified position from the same row statistics (one streaming pass
// for both)
// ---------------------------------------------------------------------------
extern "C" int dspark_verify_rates(const void* target_logits, const void* draft_logits,
                                   const int32_t* draft_tokens, const int32_t* verify_len,
                                   const float* uniforms, float temperature, int32_t dtype,
                                   int32_t B, int32_t gamma, int32_t V,
                                   const int64_t* target_row_off, const int64_t* draft_row_off,
                                   int32_t* accepted_len, int32_t* emitted_tokens,
                                   float* probs_out, uint32_t* near_tie_count, float* rates,
                                   int32_t* device_status, void* workspace,
                                   size_t workspace_bytes, struct CUstream_st* stream) {
  using namespace dspark;
  if (B > 0 && !rates) return DSPARK_ERR_INVALID_ARG;
  if (B >= 0 && B <= 65535 && gamma >= 1 && gamma <= DSPARK_MAX_GAMMA && V >= 1 &&
      V <= (1 << 30) && workspace_bytes < DSPARK_ACCEPTANCE_WS_BYTES(B, gamma, V))
    return DSPARK_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int rc = verify_entry(target_logits, draft_logits, draft_tokens, verify_len, uniforms,
                              temperature, dtype, B, gamma, V, target_row_off, draft_row_off,
                              accepted_len, emitted_tokens, probs_out, near_tie_count,
                              device_status, workspace, workspace_bytes, s, nullptr);
  if (rc != DSPARK_OK || B == 0) return rc;
  const size_t esz = dtype == DSPARK_BF16 ? 2 : 4;
  const bool aligned = (static_cast<size_t>(V) * esz) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(target_logits) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(draft_logits) % 16 == 0;
  if (dtype == DSPARK_BF16)
    return launch_rates<uint16_t>(static_cast<const uint16_t*>(target_logits),
                                  static_cast<const uint16_t*>(draft_logits), B, gamma, V,
                                  temperature, rates, device_status, workspace, s, aligned);
  return launch_rates<float>(static_cast<const float*>(target_logits),
                             static_cast<const float*>(draft_logits), B, gamma, V, temperature,
                             rates, device_status, workspace, s, aligned);
}
