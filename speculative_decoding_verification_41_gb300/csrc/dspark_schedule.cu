// dspark_schedule.cu -- hardware-aware prefix scheduler on GB300 (sm_103a).
//
// Method: "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation", section 3.2.2, and Algorithm 1 of the
// Chinese translation page: prefix survival a_{r,j} = prod_{i<=j} c_{r,i}, a
// global descending sort of the candidates with a > 0, greedy admission along
// that order with Theta = tau * SPS(B) (SPS = 1/T), stop at the first
// Theta <= Theta_best.
//
// Up to 6,144 candidates (two launches, the rank path):
//   k_sched_rank   every CTA forms all survival products a_{r,j} in shared
//                  memory (multiplied left to right in double: bit-identical to
//                  a sequential evaluation) and computes the global rank of a
//                  block of 32 candidates: each warp binary-searches a share of
//                  the requests' runs, which are already sorted because a is
//                  non-increasing in j. The order is a descending, equal values
//                  in flattened order r*gamma + j, compared as the 64-bit
//                  patterns of the doubles (exact for non-negative doubles,
//                  and integer compares: GB300's double-precision rate is about
//                  1/64 of its float rate).
//   k_sched_sweep  one CTA: tau(n) = R + sum of the n largest a in float-float
//                  (about 48 bits), the first n with Theta(n) <= Theta(n-1),
//                  compared by cross-multiplication tau(n) T(R+n-1) vs
//                  tau(n-1) T(R+n) -- every earlier step improved, so
//                  Theta_best = Theta(n-1) there -- and l_r = the largest j
//                  among the first n* candidates of request r. The decisions
//                  equal the quotient comparisons of the definition outside
//                  the 1e-9 near-tie window, which is counted.
// Beyond that (four launches, the block path): the products and a sort of
// each block of 1,024 candidates, every candidate ranked against the other
// sorted blocks, the same sweep over tiles of 4,096 positions, and the
// lengths from the ranks (k_sched_blocks, k_sched_merge, k_sched_sweep_tiled,
// k_sched_lengths). The rank path's work grows with candidates x requests,
// the block path's with candidates x blocks.
#include <climits>
#include <cmath>
#include <mutex>

#include "dspark_common.cuh"

namespace dspark {


typedef unsigned long long u64;

// Per-thread asynchronous 8-byte copy global -> shared (both addresses
// 8-byte aligned), completing with the thread's commit groups.
__device__ __forceinline__ void cp_async8(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(smem_dst)), "l"(gsrc)
               : "memory");
}

struct SchedWs {
  uint32_t* ties_scratch;
  uint32_t* n_cand;  // block path: the number of candidates (a > 0)
  int32_t* n_star;   // block path: the admitted count
  u64* keysA;  // bit patterns of non-negative doubles
  u64* keysB;
  int32_t* idxA;
  int32_t* idxB;
  int32_t* ell;
};

// Scheduling modes shared by both sweeps:
//   kModeStop     Algorithm 1: stop at the first Theta(n) <= Theta(n-1)
//   kModeGlobal   section 5.2: no break; n* = the first maximum of Theta(n)
//                 over n = 0..|E| (the capacity K of the next steps)
//   kModeTopK     section 5.2: admit the first min(K, |E|) candidates, K read
//                 from device memory
enum { kModeStop = 0, kModeGlobal = 1, kModeTopK = 2 };

// R as a float pair, exactly (R < 2^30: the low part is a small integer).
__device__ __forceinline__ ff ff_of_int(int R) {
  const float hi = static_cast<float>(R);
  return ff{hi, static_cast<float>(R - static_cast<int>(hi))};
}

__device__ __forceinline__ double d_of(const ff& x) { return static_cast<double>(x.hi) + x.lo; }

// A positive double as a float by its bits (truncated: relative error below
// 2^-23); false outside the float's normal range.
__device__ __forceinline__ bool f_of(double x, float& f) {
  const u64 b = static_cast<u64>(__double_as_longlong(x));
  const int e = static_cast<int>((b >> 52) & 0x7FF) - 1023;
  if (e < -126 || e > 127) return false;
  f = __uint_as_float((static_cast<uint32_t>(e + 127) << 23) |
                      static_cast<uint32_t>((b >> 29) & 0x7FFFFFull));
  return true;
}

// A prefix of the sorted candidates as a point of the global search:
// Theta = tau / t with t = T(R + m); m < 0 marks "none".
struct Cand {
  ff tau;
  double t;
  int m;
};

// Theta(b) > Theta(a), by cross-multiplication (both t are positive). The two
// products are formed in float from the pairs' high parts and the t's bits
// (each within 2^-22 of the double products); more than 4e-6 apart they
// decide, otherwise the double products do. Inf and NaN fail the float test.
__device__ __forceinline__ bool theta_greater(const Cand& b, const Cand& a) {
  float ta, tb;
  if (f_of(a.t, ta) && f_of(b.t, tb)) {
    const float L = b.tau.hi * ta, Rr = a.tau.hi * tb;
    if (fabsf(L - Rr) > 4e-6f * (L + Rr)) return L > Rr;
  }
  return d_of(b.tau) * a.t > d_of(a.tau) * b.t;
}

// |Theta(c) - Theta(run)| <= eps Theta(run), multiplied through by both t;
// settled in float when the products are clearly apart, as above.
__device__ __forceinline__ bool theta_tie(const Cand& c, const Cand& run) {
  float tc, tr;
  if (f_of(c.t, tc) && f_of(run.t, tr)) {
    const float L = c.tau.hi * tr, Rr = run.tau.hi * tc;
    if (fabsf(L - Rr) > 4e-6f * (L + Rr) + 1.0001e-9f * Rr) return false;
  }
  const double rt = d_of(run.tau);
  return fabs(d_of(c.tau) * run.t - rt * c.t) <= DSPARK_SCHED_TIE_REL * rt * c.t;
}

// a precedes b in the sorted order; the first maximum of Theta wins
__device__ __forceinline__ Cand cand_pick(const Cand& a, const Cand& b) {
  if (b.m < 0) return a;
  if (a.m < 0) return b;
  return theta_greater(b, a) ? b : a;
}

__device__ __forceinline__ Cand shfl_up_cand(const Cand& v, int o) {
  return Cand{ff{__shfl_up_sync(0xFFFFFFFFu, v.tau.hi, o), __shfl_up_sync(0xFFFFFFFFu, v.tau.lo, o)},
              __shfl_up_sync(0xFFFFFFFFu, v.t, o), __shfl_up_sync(0xFFFFFFFFu, v.m, o)};
}

// Exclusive scan of v over the block in thread order under cand_pick (sh: 32
// slots of shared memory). Every thread must call it.
__device__ Cand block_excl_pick(const Cand& v, Cand* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Cand none{ff{0.f, 0.f}, 1.0, -1};
  Cand incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const Cand t = shfl_up_cand(incl, o);
    if (lane >= o) incl = cand_pick(t, incl);
  }
  Cand ex = shfl_up_cand(incl, 1);
  if (lane == 0) ex = none;
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    Cand w = lane < static_cast<int>(blockDim.x >> 5) ? sh[lane] : none;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const Cand t = shfl_up_cand(w, o);
      if (lane >= o) w = cand_pick(t, w);
    }
    sh[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const Cand before = warp > 0 ? sh[warp - 1] : none;
  const Cand r = cand_pick(before, ex);
  __syncthreads();  // sh is free again
  return r;
}

// ---------------------------------------------------------------------------
// Parallel path (up to kRankMaxN candidates): ranks over the whole GPU, then a
// one-CTA sweep in float-float arithmetic.
// ---------------------------------------------------------------------------
constexpr int kRankMaxN = 6144;    // candidates of the rank path (above: the block path)
constexpr int kRankThreads = 1024;
// keys of R runs at an odd stride (within this for every batch of the rank path)
constexpr int kRankSmemMax = 196608;

// float -> double without the double-precision pipe (exact: both are IEEE
// binary formats, the double has room for every float). Zero and subnormal
// inputs take the conversion instruction.
__device__ __forceinline__ double f2d_exact(float f) {
  const uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0u || (u & 0x80000000u)) return static_cast<double>(f);
  const u64 bits = (static_cast<u64>(((u >> 23) & 0xFFu) + (1023u - 127u)) << 52) |
                   (static_cast<u64>(u & 0x7FFFFFu) << 29);
  return __longlong_as_double(static_cast<long long>(bits));
}

// A positive double's top 47 bits as a float pair, by bit manipulation. `ok`
// turns false above the float range (the caller then decides in double
// precision); values below 2^-126 read as 0.
__device__ __forceinline__ ff ff_from_bits(u64 b, bool& ok) {
  const int E = static_cast<int>((b >> 52) & 0x7FF);
  if (E == 0) {  // zero (subnormal doubles are below any value that matters here)
    if (b != 0ull) ok = false;
    return ff{0.f, 0.f};
  }
  const int e = E - 1023;
  if (e < -126) return ff{0.f, 0.f};  // below 1e-38: absorbed by any tau >= 1, as in double
  if (e > 127) {
    ok = false;
    return ff{0.f, 0.f};
  }
  const float hi = __uint_as_float((static_cast<uint32_t>(e + 127) << 23) |
                                   static_cast<uint32_t>((b >> 29) & 0x7FFFFFull));
  const float lo = ldexpf(static_cast<float>(static_cast<uint32_t>(b & 0x1FFFFFFFull)), e - 52);
  return ff{hi, lo};
}

__device__ __forceinline__ ff ff_from_double(double x, bool& ok) {
  return ff_from_bits(static_cast<u64>(__double_as_longlong(x)), ok);
}

// Survival products of every request, bit-identical to a left-to-right double
// evaluation, into keys[r * stride + j] (64-bit patterns). Returns true if a
// confidence was outside [0, 1] (it is then taken as 0).
__device__ bool survival_keys(const float* __restrict__ conf, int R, int gamma, u64* keys,
                              int stride) {
  bool bad = false;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    float cv[DSPARK_MAX_GAMMA];
#pragma unroll
    for (int j = 0; j < DSPARK_MAX_GAMMA; ++j)
      cv[j] = j < gamma ? conf[static_cast<long long>(r) * gamma + j] : 0.f;
    double prod = 1.0;
#pragma unroll
    for (int j = 0; j < DSPARK_MAX_GAMMA; ++j) {
      if (j >= gamma) break;
      float c = cv[j];
      if (!(c >= 0.f && c <= 1.f)) {
        bad = true;
        c = 0.f;
      }
      if (c == 0.f) c = 0.f;  // -0 is in [0, 1]; its product -0 would read as the largest key
      prod *= f2d_exact(c);
      keys[r * stride + j] = static_cast<u64>(__double_as_longlong(prod));
    }
  }
  return bad;
}

// Ranks of the candidates in the global order (a descending, equal values in
// flattened order). Every CTA builds all keys in shared memory once, then takes
// blocks of 32 candidates (one per lane); its 32 warps split the requests, and
// all lanes of a warp binary-search the same request's sorted run (a run of 16
// keys spans the 32 banks once: no conflicts). Partial counts merge through
// shared-memory atomics. CTA 0 also validates the inputs and writes the status.
__global__ void __launch_bounds__(kRankThreads, 1)
    k_sched_rank(const float* __restrict__ conf, int R, int gamma, SchedWs gws,
                 int32_t* status) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char smem[];
  u64* keys = reinterpret_cast<u64*>(smem);
  __shared__ int sh_bad;
  __shared__ int sh_cnt[32];
  const int n = R * gamma;
  // an odd run stride (in 8-byte keys) keeps a warp's writes of one position
  // of 32 runs within 2-way bank conflicts
  const int stride = gamma | 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int warps = blockDim.x >> 5;
  if (threadIdx.x == 0) sh_bad = 0;
  __syncthreads();
  if (survival_keys(conf, R, gamma, keys, stride)) atomicOr(&sh_bad, 1);
  __syncthreads();
  // the confidences' verdict; k_sched_sweep adds the profile's
  if (blockIdx.x == 0 && threadIdx.x == 0) *status = sh_bad ? DSPARK_ERR_BAD_DATA : DSPARK_OK;

  const int n_blocks = (n + 31) / 32;
  for (int blk = blockIdx.x; blk < n_blocks; blk += gridDim.x) {
    if (threadIdx.x < 32) sh_cnt[threadIdx.x] = 0;
    __syncthreads();
    const int e = blk * 32 + lane;
    const bool live = e < n;
    const int r = live ? e / gamma : -1;
    const int j = live ? e - r * gamma : 0;
    const u64 x = live ? keys[r * stride + j] : 0ull;
    int cnt = 0;
    for (int rr = warp; rr < R; rr += warps) {
      if (rr == r) {
        cnt += j;  // own run: the j elements before it come first (stable)
        continue;
      }
      const u64* run = keys + rr * stride;
      const bool earlier = rr < r;  // earlier request: ties come first
      int lo = 0, hi = gamma;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const u64 y = run[mid];
        if (y > x || (earlier && y == x)) lo = mid + 1; else hi = mid;
      }
      cnt += lo;
    }
    atomicAdd(&sh_cnt[lane], cnt);
    __syncthreads();
    if (warp == 0 && live) {
      const int rank = sh_cnt[lane];
      gws.keysB[rank] = x;
      gws.idxB[rank] = e;
    }
    __syncthreads();
  }
}

// The early-stop comparison of admission m: improve = tau(m) T(R+m-1) >
// tau(m-1) T(R+m), tie = the two within the near-tie window. Most admissions
// are settled in float: D = a T(R+m-1) - tau(m-1) (T(R+m) - T(R+m-1)), whose
// distance from the float-float evaluation is at most E (the float roundings,
// the dropped low parts, that evaluation's own error: E keeps a factor of ten
// over their sum); beyond E from zero and from the window's edge the two agree
// (same sign, no tie). The rest take the float-float evaluation, and values
// outside the float range double precision.
__device__ __forceinline__ void stop_compare(const ff& tau_prev, const ff& av, const ff& tau_m,
                                             const ff& tp, const ff& tm, bool okv, double Tp,
                                             double Tm, bool& improve, bool& tie) {
  if (okv) {
    const float dT = (tm.hi - tp.hi) + (tm.lo - tp.lo);
    const float A = av.hi * tp.hi, B = tau_prev.hi * dT;
    const float D = A - B;
    const float scale = tau_prev.hi * tm.hi;
    const float E = 4e-6f * (fabsf(A) + fabsf(B)) + 1e-12f * scale;
    if (fabsf(D) > E + 1.0001e-9f * scale) {  // false for inf or NaN
      improve = D > 0.f;
      tie = false;
      return;
    }
    const ff lhs = ff_mul(tau_m, tp), rhs = ff_mul(tau_prev, tm);
    improve = ff_cmp(lhs, rhs) > 0;
    const ff d = ff_sub(lhs, rhs);
    tie = fabsf(d.hi) <= static_cast<float>(DSPARK_SCHED_TIE_REL) * rhs.hi;
  } else {  // values outside the float range: double precision
    const double A = static_cast<double>(tau_m.hi) + tau_m.lo;
    const double Bv = static_cast<double>(tau_prev.hi) + tau_prev.lo;
    improve = A * Tp > Bv * Tm;
    tie = fabs(A * Tp - Bv * Tm) <= DSPARK_SCHED_TIE_REL * Bv * Tm;
  }
}

constexpr int kSweepSmemMax = (kRankMaxN + 1) * 8 + kRankMaxN * 4;  // profile slice + lengths

// Sweep over the sorted candidates (one CTA): tau(n) = R + sum of the n
// largest a in float-float, the first n whose Theta(n) = tau(n)/T(R+n) does
// not exceed Theta(n-1) (compared as tau(n) T(R+n-1) vs tau(n-1) T(R+n)),
// near ties of the evaluated comparisons, and the admitted lengths. Each
// thread owns a contiguous chunk (at most CHUNK) of the sorted order and loads its keys once,
// up front; the profile slice T(R..R(gamma+1)) is staged in shared memory and
// checked (positive, finite) on the way.
template <int CHUNK, int MODE>
__global__ void __launch_bounds__(kRankThreads, 1)
    k_sched_sweep(const double* __restrict__ T, int R, int gamma, SchedWs gws,
                  int32_t* __restrict__ verify_len, double* theta_out, uint32_t* ties,
                  int32_t* status, const int32_t* K_in, int32_t* K_out) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char smem[];
  const int n = R * gamma;
  double* sh_T = reinterpret_cast<double*>(smem);                       // T(R + m), m = 0..n
  int* sh_ell = reinterpret_cast<int*>(smem + (static_cast<size_t>(n) + 1) * 8);  // [R]
  __shared__ ff sh_w[32];
  __shared__ int sh_nE, sh_break;
  __shared__ unsigned sh_ties;
  __shared__ ff sh_tau_star;
  __shared__ Cand sh_cand[32];
  __shared__ int sh_nstar;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = (n + blockDim.x - 1) / blockDim.x;
  const int c0 = min(tid * chunk, n), c1 = min(c0 + chunk, n);
  const int len = c1 - c0;

  // every global load of the kernel is issued here, before any is waited
  // for: the profile slice by asynchronous copies, this thread's sorted values
  // and the flattened indices of its share of the order (for the lengths)
  if (T)  // the top-K admission may run without a profile
    for (int m = tid; m <= n; m += blockDim.x) cp_async8(&sh_T[m], T + R + m);
  cp_async_commit();
  u64 kv[CHUNK];
#pragma unroll
  for (int q = 0; q < CHUNK; ++q) kv[q] = q < len ? gws.keysB[c0 + q] : 0ull;
  int32_t ids[CHUNK];
#pragma unroll
  for (int k = 0; k < CHUNK; ++k) {
    const int i = tid + k * static_cast<int>(blockDim.x);
    ids[k] = i < n ? gws.idxB[i] : 0;
  }
  cp_async_wait<0>();
  bool bad_t = false;
  if (T)
    for (int m = tid; m <= n; m += blockDim.x) {
      const u64 b = static_cast<u64>(__double_as_longlong(sh_T[m]));
      if ((b >> 63) || ((b >> 52) & 0x7FFull) == 0x7FFull || b == 0ull) bad_t = true;
    }
  if (bad_t) set_status(status, DSPARK_ERR_BAD_DATA);
  if (tid == 0) {
    sh_nE = 0;
    sh_break = INT_MAX;
    sh_ties = 0;
    sh_tau_star = ff_of_int(R);
  }
  for (int r = tid; r < R; r += blockDim.x) sh_ell[r] = 0;

  // candidates: the non-zero keys, which sort first; this chunk's sum
  int cnt = 0;
  bool ok = true;
  ff local{0.f, 0.f};
#pragma unroll
  for (int q = 0; q < CHUNK; ++q) {
    cnt += kv[q] != 0ull;
    local = ff_add(local, ff_from_bits(kv[q], ok));
  }
  cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
  // exclusive block scan of the chunk sums
  ff v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff t = shfl_up_ff(v, o);
    if (lane >= o) v = ff_add(t, v);
  }
  ff ex = shfl_up_ff(v, 1);
  if (lane == 0) ex = ff{0.f, 0.f};
  __syncthreads();  // shared state initialised
  if (lane == 0) atomicAdd(&sh_nE, cnt);
  if (lane == 31) sh_w[warp] = v;
  __syncthreads();
  if (warp == 0) {
    ff w = lane < static_cast<int>(blockDim.x >> 5) ? sh_w[lane] : ff{0.f, 0.f};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const ff t = shfl_up_ff(w, o);
      if (lane >= o) w = ff_add(t, w);
    }
    sh_w[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int nE = sh_nE;
  ff tau_start = ff_add(ff_of_int(R), ex);
  if (warp > 0) tau_start = ff_add(tau_start, sh_w[warp - 1]);

  int n_star;
  if constexpr (MODE == kModeStop) {
    // walk the chunk: first non-improving admission, near ties up to it
    int first = INT_MAX;
    unsigned n_ties = 0;
    ff tau_prev = tau_start;
    bool okt = true;
    ff tp = ff_from_double(sh_T[c0], okt);
#pragma unroll
    for (int q = 0; q < CHUNK; ++q) {
      const int m = c0 + q + 1;
      if (q < len && m <= nE && first == INT_MAX) {
        bool okv = ok && okt;
        const ff av = ff_from_bits(kv[q], okv);
        const ff tau_m = ff_add(tau_prev, av);
        const double Tp = sh_T[m - 1], Tm = sh_T[m];
        const ff tm = ff_from_double(Tm, okv);
        bool improve, tie;
        stop_compare(tau_prev, av, tau_m, tp, tm, okv, Tp, Tm, improve, tie);
        if (tie) ++n_ties;
        if (!improve) first = m;
        tau_prev = tau_m;
        tp = tm;
      }
    }
    const int fw = __reduce_min_sync(0xFFFFFFFFu, first);
    if (lane == 0) atomicMin(&sh_break, fw);
    __syncthreads();
    const int n_break = sh_break;
    n_star = n_break <= nE ? n_break - 1 : nE;
    if (c0 + 1 <= n_break && n_ties) atomicAdd(&sh_ties, n_ties);
  } else if constexpr (MODE == kModeGlobal) {
    // the best admission of this chunk, then the running best before every
    // position (first maximum; position 0, nothing admitted, leads)
    Cand loc{ff{0.f, 0.f}, 1.0, -1};
    ff tau_m = tau_start;
#pragma unroll
    for (int q = 0; q < CHUNK; ++q) {
      const int m = c0 + q + 1;
      if (q < len && m <= nE) {
        bool okv = true;
        tau_m = ff_add(tau_m, ff_from_bits(kv[q], okv));
        loc = cand_pick(loc, Cand{tau_m, sh_T[m], m});
      }
    }
    Cand run = cand_pick(Cand{ff_of_int(R), sh_T[0], 0}, block_excl_pick(loc, sh_cand));
    unsigned n_ties = 0;
    tau_m = tau_start;
#pragma unroll
    for (int q = 0; q < CHUNK; ++q) {
      const int m = c0 + q + 1;
      if (q < len && m <= nE) {
        bool okv = true;
        tau_m = ff_add(tau_m, ff_from_bits(kv[q], okv));
        const Cand c{tau_m, sh_T[m], m};
        if (theta_tie(c, run)) ++n_ties;  // |Theta(m) - Theta_best| <= eps Theta_best
        run = cand_pick(run, c);
      }
    }
    n_ties = warp_sum_u32(n_ties);
    if (lane == 0 && n_ties) atomicAdd(&sh_ties, n_ties);
    if (tid == blockDim.x - 1) sh_nstar = run.m;  // the last chunk's run covers every position
    __syncthreads();
    n_star = sh_nstar;
  } else {
    int K = *K_in;
    if (K < 0) {
      if (tid == 0) set_status(status, DSPARK_ERR_BAD_DATA);
      K = 0;
    }
    n_star = K < nE ? K : nE;
  }
  // tau(n*) for Theta_best, from the thread whose chunk holds position n*
  if (n_star > 0 && c0 < n_star && n_star <= c1) {
    ff t = tau_start;
    bool okv = true;
#pragma unroll
    for (int q = 0; q < CHUNK; ++q)
      if (c0 + q < n_star) t = ff_add(t, ff_from_bits(kv[q], okv));
    sh_tau_star = t;
  }
#pragma unroll
  for (int k = 0; k < CHUNK; ++k)
    if (tid + k * static_cast<int>(blockDim.x) < n_star)
      atomicMax(&sh_ell[ids[k] / gamma], ids[k] % gamma + 1);
  __syncthreads();
  for (int r = tid; r < R; r += blockDim.x) verify_len[r] = sh_ell[r];
  if (tid == 0) {
    if (ties) *ties = sh_ties;
    if (theta_out && T) {
      const double tau_star = static_cast<double>(sh_tau_star.hi) + sh_tau_star.lo;
      *theta_out = tau_star / sh_T[n_star];
    }
    if (K_out) *K_out = n_star;
  }
}

// ---------------------------------------------------------------------------
// Block path (any number of candidates; taken above 6,144 candidates, where
// searching every request's run costs more than these four launches, and
// wherever the rank path's shared memory does not hold every key):
//   k_sched_blocks       one CTA per 1,024 candidates in flattened order: the
//                        survival products of the requests overlapping them,
//                        then a stable descending merge sort of the block.
//   k_sched_merge        one CTA per block: a candidate's rank is its place in
//                        its own block plus, for every other block, the number
//                        of that block's candidates before it (binary search;
//                        the other blocks pass through a ring of shared-memory
//                        stages filled by asynchronous copies, four blocks per
//                        step). The keys land at their ranks, and the rank of
//                        every flattened index is kept for the lengths.
//   k_sched_sweep_tiled  one CTA: the sweep of k_sched_sweep over tiles of
//                        4,096 positions (the next tile copied in while the
//                        current one is walked), stopping at the tile that
//                        holds the first non-improving admission.
//   k_sched_lengths      l_r = the number of request r's candidates whose
//                        rank is below n*.
// ---------------------------------------------------------------------------
constexpr int kBlockKeys = 1024;
constexpr int kMergeGroup = 4;                           // blocks searched per step
constexpr int kMergeGroups = 3;                          // steps in flight
constexpr int kMergeSmem = kMergeGroup * kMergeGroups * kBlockKeys * 8;  // 96 KB
constexpr int kTilePer = 4;                              // positions per thread per tile
constexpr int kSweepTile = kTilePer * kRankThreads;      // 4,096
// two tiles of sorted values and of the profile slice
constexpr int kTiledSmem = 2 * kSweepTile * 8 + 2 * (kSweepTile + 1) * 8;
constexpr int kLengthThreads = 256;

// Blocks of kBlockKeys candidates (flattened index e = r*gamma + j): CTA b
// forms a_{r,j} for the requests overlapping [b*1024, b*1024 + 1024), left to
// right in double as everywhere, and sorts the block descending, equal values
// in flattened order (a bottom-up merge: an element of a left run goes after
// the right run's strictly larger values, one of a right run after the left
// run's larger or equal ones). A request's own values never increase, so
// with gamma a power of two the merge starts from the requests' runs. Writes
// the sorted block (keys and flattened indices), a flag per request for a
// confidence outside [0, 1] (from the block holding the request's first
// candidate), and -- CTA 0 -- the status and the candidate counter.
__global__ void __launch_bounds__(kBlockKeys, 1)
    k_sched_blocks(const float* __restrict__ conf, int R, int gamma, SchedWs gws,
                   int32_t* status) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  __shared__ u64 sh_k[2][kBlockKeys];
  __shared__ int32_t sh_i[2][kBlockKeys];
  const int n = R * gamma;
  const int tid = threadIdx.x;
  const int e0 = blockIdx.x * kBlockKeys;
  const int m = min(kBlockKeys, n - e0);
  if (blockIdx.x == 0 && tid == 0) {
    *status = DSPARK_OK;
    *gws.n_cand = 0u;
  }
  const int r_first = e0 / gamma, r_last = (e0 + m - 1) / gamma;
  for (int r = r_first + tid; r <= r_last; r += kBlockKeys) {
    float cv[DSPARK_MAX_GAMMA];
#pragma unroll
    for (int j = 0; j < DSPARK_MAX_GAMMA; ++j)
      cv[j] = j < gamma ? conf[static_cast<long long>(r) * gamma + j] : 0.f;
    bool bad = false;
    double prod = 1.0;
#pragma unroll
    for (int j = 0; j < DSPARK_MAX_GAMMA; ++j) {
      if (j >= gamma) break;
      float c = cv[j];
      if (!(c >= 0.f && c <= 1.f)) {
        bad = true;
        c = 0.f;
      }
      if (c == 0.f) c = 0.f;  // -0 is in [0, 1]; its product -0 would read as the largest key
      prod *= f2d_exact(c);
      const int e = r * gamma + j;
      if (e >= e0 && e < e0 + m) {
        sh_k[0][e - e0] = static_cast<u64>(__double_as_longlong(prod));
        sh_i[0][e - e0] = e;
      }
    }
    if (r * gamma >= e0) gws.ell[r] = bad ? 1 : 0;
  }
  __syncthreads();
  int src = 0;
  // runs of gamma sit at multiples of gamma (1024 is a multiple of gamma)
  const int L0 = (gamma & (gamma - 1)) == 0 ? gamma : 1;
  for (int L = L0; L < m; L <<= 1) {
    if (tid < m) {
      const u64 x = sh_k[src][tid];
      const int a0 = (tid / (2 * L)) * (2 * L);
      const int b0 = min(a0 + L, m), b1 = min(a0 + 2 * L, m);
      const u64* A = sh_k[src];
      int dst;
      if (tid < b0) {
        int lo = b0, hi = b1;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (A[mid] > x) lo = mid + 1; else hi = mid;
        }
        dst = tid + (lo - b0);
      } else {
        int lo = a0, hi = b0;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (A[mid] >= x) lo = mid + 1; else hi = mid;
        }
        dst = a0 + (tid - b0) + (lo - a0);
      }
      sh_k[src ^ 1][dst] = x;
      sh_i[src ^ 1][dst] = sh_i[src][tid];
    }
    __syncthreads();
    src ^= 1;
  }
  if (tid < m) {
    gws.keysA[e0 + tid] = sh_k[src][tid];
    gws.idxA[e0 + tid] = sh_i[src][tid];
  }
}

// Global ranks from the sorted blocks: block o < b holds smaller flattened
// indices, so its values equal to x come first; block o > b contributes only
// its larger values. Each CTA also checks a share of the requests' flags and
// of the profile slice T(R..R(gamma+1)) (positive, finite), and adds its
// block's candidates (a > 0) to the counter.
__global__ void __launch_bounds__(kBlockKeys, 1)
    k_sched_merge(const double* __restrict__ T, int R, int gamma, SchedWs gws,
                  int32_t* status) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char smem[];
  u64* ring = reinterpret_cast<u64*>(smem);  // [kMergeGroups * kMergeGroup][kBlockKeys]
  const int n = R * gamma;
  const int nb = (n + kBlockKeys - 1) / kBlockKeys;
  const int b = blockIdx.x, tid = threadIdx.x;
  bool bad = false;
  for (long long r = static_cast<long long>(b) * kBlockKeys + tid; r < R;
       r += static_cast<long long>(nb) * kBlockKeys)
    if (__ldcg(gws.ell + r)) bad = true;
  if (T)
    for (long long m = static_cast<long long>(b) * kBlockKeys + tid; m <= n;
         m += static_cast<long long>(nb) * kBlockKeys) {
      const u64 t = static_cast<u64>(__double_as_longlong(T[R + m]));
      if ((t >> 63) || ((t >> 52) & 0x7FFull) == 0x7FFull || t == 0ull) bad = true;
    }
  if (bad) set_status(status, DSPARK_ERR_BAD_DATA);

  const int e0 = b * kBlockKeys;
  const int mine = min(kBlockKeys, n - e0);
  const bool live = tid < mine;
  const u64 x = live ? __ldcg(gws.keysA + e0 + tid) : 0ull;
  const int id = live ? __ldcg(gws.idxA + e0 + tid) : 0;
  const int cand = __syncthreads_count(live && x != 0ull);
  if (tid == 0 && cand) atomicAdd(gws.n_cand, static_cast<uint32_t>(cand));

  // the other blocks in visiting order: visit q is block q, or q + 1 from this
  // block on; step s searches visits [s*G, s*G + G)
  const int others = nb - 1;
  const int steps = (others + kMergeGroup - 1) / kMergeGroup;
  auto issue = [&](int s) {
    if (s < steps) {
      for (int g = 0; g < kMergeGroup; ++g) {
        const int q = s * kMergeGroup + g;
        if (q >= others) break;
        const int o = q + (q >= b);
        const int len = min(kBlockKeys, n - o * kBlockKeys);
        const u64* srcp = gws.keysA + static_cast<size_t>(o) * kBlockKeys;
        u64* dst = ring + static_cast<size_t>((s % kMergeGroups) * kMergeGroup + g) * kBlockKeys;
        for (int v = tid; v < len / 2; v += kBlockKeys) cp_async16(dst + 2 * v, srcp + 2 * v);
        if ((len & 1) && tid == 0) cp_async8(dst + len - 1, srcp + len - 1);
        // a short (last) block is padded with zeros, which no candidate counts
        for (int v = len + tid; v < kBlockKeys; v += kBlockKeys) dst[v] = 0ull;
      }
    }
    cp_async_commit();  // empty groups complete at once
  };
#pragma unroll
  for (int s = 0; s < kMergeGroups - 1; ++s) issue(s);
  int rank = tid;
  for (int s = 0; s < steps; ++s) {
    issue(s + kMergeGroups - 1);  // the stages read at s - 1, released by its barrier
    cp_async_wait<kMergeGroups - 1>();
    __syncthreads();  // every thread's copies of step s have landed
    if (live && x != 0ull) {
      // per block, the number of its values >= x (earlier blocks: equal
      // values come first) or >= x + 1 (later blocks); the keys are integers,
      // the blocks descending and zero-padded to 1024, so a 10-step lift
      // finds each count; the group's lifts run side by side
      int pos[kMergeGroup];
      u64 xq[kMergeGroup];
      const u64* run[kMergeGroup];
#pragma unroll
      for (int g = 0; g < kMergeGroup; ++g) {
        const int q = s * kMergeGroup + g;
        pos[g] = 0;
        xq[g] = q >= others ? ~0ull : (q < b ? x : x + 1ull);  // past the end: counts nothing
        run[g] = ring + static_cast<size_t>((s % kMergeGroups) * kMergeGroup + g) * kBlockKeys;
      }
#pragma unroll
      for (int step = kBlockKeys / 2; step >= 1; step >>= 1)
#pragma unroll
        for (int g = 0; g < kMergeGroup; ++g)
          pos[g] += run[g][pos[g] + step - 1] >= xq[g] ? step : 0;
#pragma unroll
      for (int g = 0; g < kMergeGroup; ++g)
        rank += pos[g] + (pos[g] == kBlockKeys - 1 && run[g][kBlockKeys - 1] >= xq[g]);
    }
    __syncthreads();  // step s's stages may be refilled
  }
  cp_async_wait<0>();
  if (live) {
    // the candidates (a > 0) take ranks 0..|E|-1 and their values land there;
    // a zero value is no candidate: its rank only has to exceed any n*
    if (x != 0ull) gws.keysB[rank] = x;
    gws.idxB[id] = x != 0ull ? rank : INT_MAX;  // the rank of flattened index id
  }
}

// The sweep of k_sched_sweep (same float-float arithmetic, comparisons and
// near-tie counts) over tiles of kSweepTile positions, with tau and, for the
// global search, the best admission so far carried from tile to tile; each
// tile's sorted values and profile slice are copied into shared memory while
// the one before is walked. The profile slice was checked by k_sched_merge.
// Writes n* to the workspace header for k_sched_lengths.
template <int MODE>
__global__ void __launch_bounds__(kRankThreads, 1)
    k_sched_sweep_tiled(const double* __restrict__ T, int R, int gamma, SchedWs gws,
                        double* theta_out, uint32_t* ties, int32_t* status,
                        const int32_t* K_in, int32_t* K_out) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char smem[];
  u64* sh_key = reinterpret_cast<u64*>(smem);                                  // [2][kSweepTile]
  double* sh_Tb = reinterpret_cast<double*>(smem + 2 * kSweepTile * 8);        // [2][kSweepTile + 1]
  __shared__ ff sh_w[32];
  __shared__ int sh_break;
  __shared__ unsigned sh_ties;
  __shared__ ff sh_carry, sh_tau_star;
  __shared__ Cand sh_cand[32];
  __shared__ Cand sh_best;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nE = static_cast<int>(__ldcg(gws.n_cand));
  if (tid == 0) {
    sh_break = INT_MAX;
    sh_ties = 0;
    sh_carry = ff_of_int(R);
    sh_tau_star = ff_of_int(R);
    if (MODE == kModeGlobal) sh_best = Cand{ff_of_int(R), T[R], 0};
  }
  // tile t0's values and profile slice T(R + t0 + i), i = 0..len, into buffer p
  auto fetch = [&](int t0, int p) {
    const int len = min(kSweepTile, nE - t0);
    u64* kd = sh_key + p * kSweepTile;
    double* td = sh_Tb + p * (kSweepTile + 1);
    const u64* ks = gws.keysB + t0;  // t0 is a multiple of kSweepTile: 16-byte aligned
    for (int v = tid; v < len / 2; v += blockDim.x) cp_async16(kd + 2 * v, ks + 2 * v);
    if ((len & 1) && tid == 0) cp_async8(kd + len - 1, ks + len - 1);
    for (int i = tid; i <= len; i += blockDim.x) cp_async8(td + i, T + R + t0 + i);
    cp_async_commit();
  };
  int n_star = 0;
  if constexpr (MODE == kModeTopK) {
    __syncthreads();
    int K = *K_in;
    if (K < 0) {
      if (tid == 0) set_status(status, DSPARK_ERR_BAD_DATA);
      K = 0;
    }
    n_star = K < nE ? K : nE;
    if (theta_out && T) {  // tau(n*) over the first n* sorted values
      ff s{0.f, 0.f};
      bool okv = true;
      for (int i = tid; i < n_star; i += blockDim.x)
        s = ff_add(s, ff_from_bits(__ldcg(gws.keysB + i), okv));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        s = ff_add(s, ff{__shfl_xor_sync(0xFFFFFFFFu, s.hi, o),
                         __shfl_xor_sync(0xFFFFFFFFu, s.lo, o)});
      if (lane == 0) sh_w[warp] = s;
      __syncthreads();
      if (tid == 0) {
        ff t{static_cast<float>(R), 0.f};
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t = ff_add(t, sh_w[w]);
        sh_tau_star = t;
      }
    }
  } else {
    if (nE > 0) fetch(0, 0);
    bool stopped = false;
    int p = 0;
    for (int t0 = 0; t0 < nE && !stopped; t0 += kSweepTile, p ^= 1) {
      cp_async_wait<0>();
      __syncthreads();  // tile t0 in buffer p; buffer p ^ 1 free (its tile was walked)
      if (t0 + kSweepTile < nE) fetch(t0 + kSweepTile, p ^ 1);
      const u64* kt = sh_key + p * kSweepTile;
      const double* sh_T = sh_Tb + p * (kSweepTile + 1);
      const int lenT = min(kSweepTile, nE - t0);  // positions t0 + 1 .. t0 + lenT
      const int c0 = min(tid * kTilePer, lenT), c1 = min(c0 + kTilePer, lenT);
      const int len = c1 - c0;
      u64 kv[kTilePer];
#pragma unroll
      for (int q = 0; q < kTilePer; ++q) kv[q] = q < len ? kt[c0 + q] : 0ull;
      bool ok = true;
      ff local{0.f, 0.f};
#pragma unroll
      for (int q = 0; q < kTilePer; ++q) local = ff_add(local, ff_from_bits(kv[q], ok));
      ff v = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const ff t = shfl_up_ff(v, o);
        if (lane >= o) v = ff_add(t, v);
      }
      ff ex = shfl_up_ff(v, 1);
      if (lane == 0) ex = ff{0.f, 0.f};
      if (lane == 31) sh_w[warp] = v;
      __syncthreads();
      if (warp == 0) {
        ff w = lane < static_cast<int>(blockDim.x >> 5) ? sh_w[lane] : ff{0.f, 0.f};
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const ff t = shfl_up_ff(w, o);
          if (lane >= o) w = ff_add(t, w);
        }
        sh_w[lane] = w;  // inclusive over warps
      }
      __syncthreads();
      const ff carry = sh_carry;
      ff tau_start = ff_add(carry, ex);
      if (warp > 0) tau_start = ff_add(tau_start, sh_w[warp - 1]);

      if constexpr (MODE == kModeStop) {
        int first = INT_MAX;
        unsigned n_ties = 0;
        ff tau_prev = tau_start;
        bool okt = true;
        ff tp = ff_from_double(sh_T[c0], okt);
#pragma unroll
        for (int q = 0; q < kTilePer; ++q) {
          const int m = t0 + c0 + q + 1;
          if (q < len && first == INT_MAX) {
            bool okv = ok && okt;
            const ff av = ff_from_bits(kv[q], okv);
            const ff tau_m = ff_add(tau_prev, av);
            const double Tp = sh_T[c0 + q], Tm = sh_T[c0 + q + 1];
            const ff tm = ff_from_double(Tm, okv);
            bool improve, tie;
            stop_compare(tau_prev, av, tau_m, tp, tm, okv, Tp, Tm, improve, tie);
            if (tie) ++n_ties;
            if (!improve) first = m;
            tau_prev = tau_m;
            tp = tm;
          }
        }
        const int fw = __reduce_min_sync(0xFFFFFFFFu, first);
        if (lane == 0 && fw != INT_MAX) atomicMin(&sh_break, fw);
        __syncthreads();
        const int n_break = sh_break;
        if (t0 + c0 + 1 <= n_break && n_ties) atomicAdd(&sh_ties, n_ties);
        if (n_break != INT_MAX) {
          stopped = true;
          n_star = n_break - 1;
          // tau(n*): the tile's start when n* = t0, else from the chunk holding it
          if (n_star > t0 && t0 + c0 < n_star && n_star <= t0 + c1) {
            ff t = tau_start;
            bool okv = true;
#pragma unroll
            for (int q = 0; q < kTilePer; ++q)
              if (t0 + c0 + q < n_star) t = ff_add(t, ff_from_bits(kv[q], okv));
            sh_tau_star = t;
          } else if (n_star == t0 && tid == 0) {
            sh_tau_star = carry;
          }
        }
      } else {  // kModeGlobal
        Cand loc{ff{0.f, 0.f}, 1.0, -1};
        ff tau_m = tau_start;
#pragma unroll
        for (int q = 0; q < kTilePer; ++q) {
          if (q < len) {
            bool okv = true;
            tau_m = ff_add(tau_m, ff_from_bits(kv[q], okv));
            loc = cand_pick(loc, Cand{tau_m, sh_T[c0 + q + 1], t0 + c0 + q + 1});
          }
        }
        Cand run = cand_pick(sh_best, block_excl_pick(loc, sh_cand));
        unsigned n_ties = 0;
        tau_m = tau_start;
#pragma unroll
        for (int q = 0; q < kTilePer; ++q) {
          if (q < len) {
            bool okv = true;
            tau_m = ff_add(tau_m, ff_from_bits(kv[q], okv));
            const Cand c{tau_m, sh_T[c0 + q + 1], t0 + c0 + q + 1};
            if (theta_tie(c, run)) ++n_ties;
            run = cand_pick(run, c);
          }
        }
        n_ties = warp_sum_u32(n_ties);
        if (lane == 0 && n_ties) atomicAdd(&sh_ties, n_ties);
        __syncthreads();  // every thread has read sh_best
        if (tid == blockDim.x - 1) sh_best = run;  // the last chunk's run covers the tile
      }
      // tau after the tile, for the next one
      if (tid == blockDim.x - 1) sh_carry = ff_add(tau_start, local);
    }
    cp_async_wait<0>();  // a prefetch past the stopping tile lands before the exit
    __syncthreads();
    if (MODE == kModeStop && !stopped) {
      n_star = nE;
      if (tid == 0) sh_tau_star = sh_carry;
    }
    if (MODE == kModeGlobal) n_star = sh_best.m;
  }
  __syncthreads();
  if (tid == 0) {
    *gws.n_star = n_star;
    if (ties) *ties = sh_ties;
    if (theta_out && T) {
      if (MODE == kModeGlobal) {
        *theta_out = d_of(sh_best.tau) / sh_best.t;
      } else {
        const double tau_star = static_cast<double>(sh_tau_star.hi) + sh_tau_star.lo;
        *theta_out = tau_star / T[R + n_star];
      }
    }
    if (K_out) *K_out = n_star;
  }
}

// l_r: request r's candidates among the first n* (a prefix of its run, since
// a does not increase with j), from the ranks of its flattened indices.
__global__ void __launch_bounds__(kLengthThreads)
    k_sched_lengths(int R, int gamma, SchedWs gws, int32_t* __restrict__ verify_len) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  const int r = blockIdx.x * kLengthThreads + threadIdx.x;
  if (r >= R) return;
  const int n_star = __ldcg(gws.n_star);
  const int32_t* rk = gws.idxB + static_cast<size_t>(r) * gamma;
  int l = 0;
  for (int j0 = 0; j0 < gamma; j0 += 8) {  // eight independent loads at a time
    int32_t v[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) v[t] = j0 + t < gamma ? __ldcg(rk + j0 + t) : INT_MAX;
#pragma unroll
    for (int t = 0; t < 8; ++t) l += v[t] < n_star;
  }
  verify_len[r] = l;
}

// Static-threshold lengths (section 4.3.3, the diagnostic baseline): l_r =
// the number of leading draft tokens whose confidence reaches the threshold.
// One CTA, a thread per request; the CTA sees every confidence, so its verdict
// on them is complete when thread 0 writes the status.
__global__ void __launch_bounds__(1024, 1)
    k_sched_threshold(const float* __restrict__ conf, float thr, int R, int gamma,
                      int32_t* __restrict__ verify_len, int32_t* status) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  __shared__ int sh_bad;
  if (threadIdx.x == 0) sh_bad = 0;
  __syncthreads();
  bool bad = false;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    const float* c = conf + static_cast<long long>(r) * gamma;
    int ell = 0;
    bool open = true;
    for (int j = 0; j < gamma; ++j) {
      const float v = c[j];
      if (!(v >= 0.f && v <= 1.f)) bad = true;
      if (open && v >= thr)
        ++ell;
      else
        open = false;
    }
    verify_len[r] = ell;
  }
  if (bad) atomicOr(&sh_bad, 1);
  __syncthreads();
  if (threadIdx.x == 0) *status = sh_bad ? DSPARK_ERR_BAD_DATA : DSPARK_OK;
}

template <int MODE>
bool sweep_smem_attr() {
  return cudaFuncSetAttribute(k_sched_sweep<4, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSweepSmemMax) == cudaSuccess &&
         cudaFuncSetAttribute(k_sched_sweep<8, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSweepSmemMax) == cudaSuccess;
}

// the sweep instantiation whose per-thread chunk holds n / 1024 candidates
// (n <= kRankMaxN <= 8 * 1024)
template <int MODE>
cudaError_t launch_sweep(int n, size_t smem, cudaStream_t st, const double* T, int R, int gamma,
                         const SchedWs& ws, int32_t* verify_len, double* theta, uint32_t* ties,
                         int32_t* status, const int32_t* K_in, int32_t* K_out) {
  static_assert(kRankMaxN <= 8 * kRankThreads, "rank path larger than the sweep's chunks");
  if (n <= 4 * kRankThreads)
    return launch_pdl(k_sched_sweep<4, MODE>, 1, kRankThreads, smem, st, T, R, gamma, ws,
                      verify_len, theta, ties, status, K_in, K_out);
  return launch_pdl(k_sched_sweep<8, MODE>, 1, kRankThreads, smem, st, T, R, gamma, ws,
                    verify_len, theta, ties, status, K_in, K_out);
}

std::mutex g_sched_mutex;
bool g_sched_ready[128];
int g_sched_sms[128];

}  // namespace dspark

namespace dspark {

// Shared host path of the three scheduler entry points. T may be NULL only in
// the top-K mode (no profile, no Theta).
int schedule_run(int mode, const float* confidences, const double* step_time_ms,
                 int64_t n_profile, int32_t R, int32_t gamma, const int32_t* K_in,
                 int32_t* K_out, int32_t* verify_len, double* theta_best,
                 uint32_t* near_tie_count, int32_t* device_status, void* workspace,
                 size_t workspace_bytes, cudaStream_t st) {
  if (R < 1 || gamma < 1 || gamma > DSPARK_MAX_GAMMA) return DSPARK_ERR_INVALID_ARG;
  if (static_cast<long long>(R) * (gamma + 1) >= (1LL << 30)) return DSPARK_ERR_INVALID_ARG;
  if (!confidences || !verify_len || !device_status) return DSPARK_ERR_INVALID_ARG;
  if (mode != kModeTopK || step_time_ms) {
    if (!step_time_ms) return DSPARK_ERR_INVALID_ARG;
    if (n_profile < static_cast<int64_t>(R) * (gamma + 1) + 1) return DSPARK_ERR_INVALID_ARG;
  }
  if (mode == kModeTopK && !K_in) return DSPARK_ERR_INVALID_ARG;
  if (mode == kModeGlobal && !K_out) return DSPARK_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < DSPARK_SCHEDULE_WS_BYTES(R, gamma) ||
      reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return DSPARK_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return DSPARK_ERR_CUDA;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lock(g_sched_mutex);
    if (!g_sched_ready[dev]) {
      if (cudaFuncSetAttribute(k_sched_sweep_tiled<kModeStop>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kTiledSmem) != cudaSuccess ||
          cudaFuncSetAttribute(k_sched_sweep_tiled<kModeGlobal>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kTiledSmem) != cudaSuccess ||
          cudaFuncSetAttribute(k_sched_sweep_tiled<kModeTopK>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kTiledSmem) != cudaSuccess ||
          cudaFuncSetAttribute(k_sched_merge, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kMergeSmem) != cudaSuccess)
        return DSPARK_ERR_CUDA;
      if (cudaFuncSetAttribute(k_sched_rank, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kRankSmemMax) != cudaSuccess)
        return DSPARK_ERR_CUDA;
      if (!sweep_smem_attr<kModeStop>() || !sweep_smem_attr<kModeGlobal>() ||
          !sweep_smem_attr<kModeTopK>())
        return DSPARK_ERR_CUDA;
      if (cudaDeviceGetAttribute(&g_sched_sms[dev], cudaDevAttrMultiProcessorCount, dev) !=
          cudaSuccess)
        return DSPARK_ERR_CUDA;
      g_sched_ready[dev] = true;
    }
    sms = g_sched_sms[dev];
  }
  const int n = R * gamma;
  char* p = static_cast<char*>(workspace);
  SchedWs ws;
  ws.ties_scratch = reinterpret_cast<uint32_t*>(p);
  ws.n_cand = reinterpret_cast<uint32_t*>(p + 64);
  ws.n_star = reinterpret_cast<int32_t*>(p + 128);
  p += 256;
  ws.keysA = reinterpret_cast<u64*>(p);
  p += DSPARK_ALIGN256(static_cast<size_t>(n) * 8);
  ws.keysB = reinterpret_cast<u64*>(p);
  p += DSPARK_ALIGN256(static_cast<size_t>(n) * 8);
  ws.idxA = reinterpret_cast<int32_t*>(p);
  p += DSPARK_ALIGN256(static_cast<size_t>(n) * 4);
  ws.idxB = reinterpret_cast<int32_t*>(p);
  p += DSPARK_ALIGN256(static_cast<size_t>(n) * 4);
  ws.ell = reinterpret_cast<int32_t*>(p);
  uint32_t* ties = near_tie_count ? near_tie_count : ws.ties_scratch;
  const double* T = step_time_ms;
  const size_t rank_smem = static_cast<size_t>(R) * (gamma | 1) * 8;
  if (n <= kRankMaxN && rank_smem <= static_cast<size_t>(kRankSmemMax)) {
    // ranks over the whole GPU, then a one-CTA float-float sweep
    const int blocks = (n + 31) / 32;
    const int grid = blocks < sms ? blocks : sms;
    cudaError_t e = launch_pdl(k_sched_rank, grid, kRankThreads, rank_smem, st, confidences, R,
                               gamma, ws, device_status);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
    const size_t sweep_smem = (static_cast<size_t>(n) + 1) * 8 + static_cast<size_t>(R) * 4;
    if (mode == kModeStop)
      e = launch_sweep<kModeStop>(n, sweep_smem, st, T, R, gamma, ws, verify_len, theta_best,
                                  ties, device_status, K_in, K_out);
    else if (mode == kModeGlobal)
      e = launch_sweep<kModeGlobal>(n, sweep_smem, st, T, R, gamma, ws, verify_len, theta_best,
                                    ties, device_status, K_in, K_out);
    else
      e = launch_sweep<kModeTopK>(n, sweep_smem, st, T, R, gamma, ws, verify_len, theta_best,
                                  ties, device_status, K_in, K_out);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  } else {
    // sorted blocks, ranks against the other blocks, a tiled one-CTA sweep,
    // the lengths
    const int nb = (n + kBlockKeys - 1) / kBlockKeys;
    cudaError_t e = launch_pdl(k_sched_blocks, nb, kBlockKeys, 0, st, confidences, R, gamma, ws,
                               device_status);
    if (e == cudaSuccess)
      e = launch_pdl(k_sched_merge, nb, kBlockKeys, static_cast<size_t>(kMergeSmem), st, T, R,
                     gamma, ws, device_status);
    if (e == cudaSuccess) {
      if (mode == kModeStop)
        e = launch_pdl(k_sched_sweep_tiled<kModeStop>, 1, kRankThreads, kTiledSmem, st, T, R,
                       gamma, ws, theta_best, ties, device_status, K_in, K_out);
      else if (mode == kModeGlobal)
        e = launch_pdl(k_sched_sweep_tiled<kModeGlobal>, 1, kRankThreads, kTiledSmem, st, T, R,
                       gamma, ws, theta_best, ties, device_status, K_in, K_out);
      else
        e = launch_pdl(k_sched_sweep_tiled<kModeTopK>, 1, kRankThreads, kTiledSmem, st, T, R,
                       gamma, ws, theta_best, ties, device_status, K_in, K_out);
    }
    if (e == cudaSuccess)
      e = launch_pdl(k_sched_lengths, (R + kLengthThreads - 1) / kLengthThreads, kLengthThreads,
                     0, st, R, gamma, ws, verify_len);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}

}  // namespace dspark

extern "C" int dspark_schedule(const float* confidences, const double* step_time_ms,
                               int64_t n_profile, int32_t R, int32_t gamma, int32_t* verify_len,
                               double* theta_best, uint32_t* near_tie_count,
                               int32_t* device_status, void* workspace, size_t workspace_bytes,
                               struct CUstream_st* stream) {
  return dspark::schedule_run(dspark::kModeStop, confidences, step_time_ms, n_profile, R, gamma,
                              nullptr, nullptr, verify_len, theta_best, near_tie_count,
                              device_status, workspace, workspace_bytes,
                              reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int dspark_schedule_capacity(const float* confidences, const double* step_time_ms,
                                        int64_t n_profile, int32_t R, int32_t gamma,
                                        int32_t* capacity, int32_t* verify_len,
                                        double* theta_best, uint32_t* near_tie_count,
                                        int32_t* device_status, void* workspace,
                                        size_t workspace_bytes, struct CUstream_st* stream) {
  return dspark::schedule_run(dspark::kModeGlobal, confidences, step_time_ms, n_profile, R,
                              gamma, nullptr, capacity, verify_len, theta_best, near_tie_count,
                              device_status, workspace, workspace_bytes,
                              reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int dspark_schedule_topk(const float* confidences, const int32_t* capacity, int32_t R,
                                    int32_t gamma, int32_t* verify_len, int32_t* device_status,
                                    void* workspace, size_t workspace_bytes,
                                    struct CUstream_st* stream) {
  return dspark::schedule_run(dspark::kModeTopK, confidences, nullptr, 0, R, gamma, capacity,
                              nullptr, verify_len, nullptr, nullptr, device_status, workspace,
                              workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int dspark_schedule_threshold(const float* confidences, float threshold, int32_t R,
                                         int32_t gamma, int32_t* verify_len,
                                         int32_t* device_status, struct CUstream_st* stream) {
  using namespace dspark;
  if (R < 1 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || !std::isfinite(threshold))
    return DSPARK_ERR_INVALID_ARG;
  if (!confidences || !verify_len || !device_status) return DSPARK_ERR_INVALID_ARG;
  if (launch_pdl(k_sched_threshold, 1, 1024, 0, reinterpret_cast<cudaStream_t>(stream),
                 confidences, threshold, R, gamma, verify_len, device_status) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}
