// dspark_schedule.cu -- hardware-aware prefix scheduler on GB300 (sm_103a).
//
// Method: "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation", section 3.2.2, and Algorithm 1 of the
// Chinese translation page: prefix survival a_{r,j} = prod_{i<=j} c_{r,i}, a
// global descending sort of the candidates with a > 0, greedy admission along
// that order with Theta = tau * SPS(B) (SPS = 1/T), stop at the first
// Theta <= Theta_best.
//
// Up to 16,384 candidates (two launches):
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
// Beyond that, k_schedule does everything in one CTA: the same products, a
// merge sort of the runs (pairwise merges by rank), a double block scan and a
// double sweep.
#include <climits>
#include <cmath>
#include <mutex>

#include "dspark_common.cuh"

namespace dspark {

constexpr int kSchedThreads = 1024;
constexpr int kSchedSmemMaxN = 8192;  // candidates kept in shared memory (24 B each)

typedef unsigned long long u64;

struct SchedWs {
  uint32_t* ties_scratch;
  u64* keysA;  // bit patterns of non-negative doubles
  u64* keysB;
  int32_t* idxA;
  int32_t* idxB;
  int32_t* ell;
};

__device__ __forceinline__ double block_sum_excl(double v, double* sh, double& total) {
  // exclusive prefix of v over the block (1024 threads), and the block total
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    double w = sh[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += t;
    }
    sh[lane] = w;
  }
  __syncthreads();
  const double before = (warp ? sh[warp - 1] : 0.0) + (incl - v);
  total = sh[31];
  __syncthreads();
  return before;
}

// Scheduling modes shared by the sweep and the one-CTA path:
//   kModeStop     Algorithm 1: stop at the first Theta(n) <= Theta(n-1)
//   kModeGlobal   section 5.2: no break; n* = the first maximum of Theta(n)
//                 over n = 0..|E| (the capacity K of the next steps)
//   kModeTopK     section 5.2: admit the first min(K, |E|) candidates, K read
//                 from device memory
enum { kModeStop = 0, kModeGlobal = 1, kModeTopK = 2 };

// A prefix of the sorted candidates as a point of the global search:
// Theta = tau / t with t = T(R + m); m < 0 marks "none".
struct Cand {
  double tau, t;
  int m;
};

// a precedes b in the sorted order; the first maximum of Theta wins (compared
// by cross-multiplication: both t are positive)
__device__ __forceinline__ Cand cand_pick(const Cand& a, const Cand& b) {
  if (b.m < 0) return a;
  if (a.m < 0) return b;
  return b.tau * a.t > a.tau * b.t ? b : a;
}

__device__ __forceinline__ Cand shfl_up_cand(const Cand& v, int o) {
  return Cand{__shfl_up_sync(0xFFFFFFFFu, v.tau, o), __shfl_up_sync(0xFFFFFFFFu, v.t, o),
              __shfl_up_sync(0xFFFFFFFFu, v.m, o)};
}

// Exclusive scan of v over the block in thread order under cand_pick (sh: 32
// slots of shared memory). Every thread must call it.
__device__ Cand block_excl_pick(const Cand& v, Cand* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Cand none{0.0, 1.0, -1};
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

__global__ void __launch_bounds__(kSchedThreads, 1)
    k_schedule(const float* __restrict__ conf, const double* __restrict__ T, int R, int gamma,
               int32_t* __restrict__ verify_len, double* theta_out, uint32_t* ties,
               int32_t* status, SchedWs gws, int use_smem, int mode, const int32_t* K_in,
               int32_t* K_out) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ double red[32];
  __shared__ int red_i[32];
  __shared__ int sh_n_break, sh_nE;
  __shared__ unsigned sh_ties;
  __shared__ Cand sh_cand[32];
  __shared__ int sh_nstar;
  const int n = R * gamma;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  u64* kA = gws.keysA;
  u64* kB = gws.keysB;
  int32_t* iA = gws.idxA;
  int32_t* iB = gws.idxB;
  if (use_smem) {
    kA = reinterpret_cast<u64*>(smem);
    kB = kA + n;
    iA = reinterpret_cast<int32_t*>(kB + n);
    iB = iA + n;
  }
  if (tid == 0) {
    *status = DSPARK_OK;
    if (ties) *ties = 0;
    sh_n_break = INT_MAX;
    sh_nE = 0;
    sh_ties = 0;
  }
  __syncthreads();

  // 1. prefix survival probabilities
  for (int r = tid; r < R; r += kSchedThreads) {
    // all of the request's loads are issued before the multiply chain
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
        set_status(status, DSPARK_ERR_BAD_DATA);
        c = 0.f;
      }
      prod *= static_cast<double>(c);
      kA[r * gamma + j] = static_cast<u64>(__double_as_longlong(prod));
      iA[r * gamma + j] = r * gamma + j;
    }
    gws.ell[r] = 0;
  }
  // profile entries that can be looked up must be positive and finite
  if (T)
    for (int b = R + tid; b <= R * (gamma + 1); b += kSchedThreads)
      if (!(T[b] > 0.0) || !isfinite(T[b])) set_status(status, DSPARK_ERR_BAD_DATA);
  __syncthreads();

  // 2. stable descending merge of the per-request runs
  for (int L = gamma; L < n; L *= 2) {
    for (int i = tid; i < n; i += kSchedThreads) {
      const int a0 = (i / (2 * L)) * (2 * L);
      const int b0 = min(a0 + L, n), b1 = min(a0 + 2 * L, n);
      const u64 key = kA[i];
      int dst;
      if (i < b0) {  // left run: right-run elements strictly greater come first
        int lo = b0, hi = b1;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (kA[mid] > key) lo = mid + 1; else hi = mid;
        }
        dst = i + (lo - b0);
      } else {       // right run: left-run elements greater or equal come first
        int lo = a0, hi = b0;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (kA[mid] >= key) lo = mid + 1; else hi = mid;
        }
        dst = a0 + (i - b0) + (lo - a0);
      }
      kB[dst] = key;
      iB[dst] = iA[i];
    }
    __syncthreads();
    u64* tk = kA; kA = kB; kB = tk;
    int32_t* ti = iA; iA = iB; iB = ti;
  }

  // 3. number of candidates (a > 0 sort first) and tau(n) into kB
  {
    int cnt = 0;
    for (int i = tid; i < n; i += kSchedThreads) cnt += kA[i] != 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
    if (lane == 0) atomicAdd(&sh_nE, cnt);
  }
  __syncthreads();
  const int nE = sh_nE;
  const int chunk = (nE + kSchedThreads - 1) / kSchedThreads;
  const int c0 = min(tid * chunk, nE), c1 = min(c0 + chunk, nE);
  double local = 0.0;
  for (int i = c0; i < c1; ++i) local += __longlong_as_double(static_cast<long long>(kA[i]));
  double total;
  const double before = block_sum_excl(local, red, total);
  double run = static_cast<double>(R) + before;
  double* tau = reinterpret_cast<double*>(kB);  // tau(i + 1) in the free buffer
  for (int i = c0; i < c1; ++i) {
    run += __longlong_as_double(static_cast<long long>(kA[i]));
    tau[i] = run;
  }
  __syncthreads();

  int n_star;
  if (mode == kModeStop) {
    // 4. first non-improving admission
    int first = INT_MAX;
    for (int m = 1 + tid; m <= nE; m += kSchedThreads) {
      const double tau_m = tau[m - 1];
      const double tau_p = m == 1 ? static_cast<double>(R) : tau[m - 2];
      if (!(tau_m * T[R + m - 1] > tau_p * T[R + m])) first = min(first, m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xFFFFFFFFu, first, o));
    if (lane == 0) red_i[warp] = first;
    __syncthreads();
    if (warp == 0) {
      int f = red_i[lane];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) f = min(f, __shfl_xor_sync(0xFFFFFFFFu, f, o));
      if (lane == 0) sh_n_break = f;
    }
    __syncthreads();
    const int n_break = sh_n_break;  // INT_MAX: every admission improved
    n_star = n_break <= nE ? n_break - 1 : nE;
    // near ties among the comparisons actually evaluated (steps 1..min(n_break, nE))
    const int last = min(n_break, nE);
    unsigned t = 0;
    for (int m = 1 + tid; m <= last; m += kSchedThreads) {
      const double tau_m = tau[m - 1];
      const double tau_p = m == 1 ? static_cast<double>(R) : tau[m - 2];
      const double tm = T[R + m], tp = T[R + m - 1];
      // |Theta(m) - Theta(m-1)| <= eps Theta(m-1), multiplied through by T(R+m) T(R+m-1)
      if (fabs(tau_m * tp - tau_p * tm) <= DSPARK_SCHED_TIE_REL * tau_p * tm) ++t;
    }
    t = warp_sum_u32(t);
    if (lane == 0 && t) atomicAdd(&sh_ties, t);
  } else if (mode == kModeGlobal) {
    // 4'. first maximum of Theta over n = 0..|E|: chunk bests, their exclusive
    // scan, then every admission against the best before it
    const int gc = (nE + kSchedThreads - 1) / kSchedThreads;
    const int g0 = min(tid * gc, nE), g1 = min(g0 + gc, nE);
    Cand loc{0.0, 1.0, -1};
    for (int m = g0 + 1; m <= g1; ++m) loc = cand_pick(loc, Cand{tau[m - 1], T[R + m], m});
    Cand run = cand_pick(Cand{static_cast<double>(R), T[R], 0}, block_excl_pick(loc, sh_cand));
    unsigned t = 0;
    for (int m = g0 + 1; m <= g1; ++m) {
      const Cand c{tau[m - 1], T[R + m], m};
      if (fabs(c.tau * run.t - run.tau * c.t) <= DSPARK_SCHED_TIE_REL * run.tau * c.t) ++t;
      run = cand_pick(run, c);
    }
    t = warp_sum_u32(t);
    if (lane == 0 && t) atomicAdd(&sh_ties, t);
    if (tid == kSchedThreads - 1) sh_nstar = run.m;  // the last chunk's run covers every position
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
  // 5. verify lengths: the admitted prefix of each request
  for (int i = tid; i < n_star; i += kSchedThreads) {
    const int id = iA[i];
    atomicMax(&gws.ell[id / gamma], id % gamma + 1);
  }
  __syncthreads();
  for (int r = tid; r < R; r += kSchedThreads) verify_len[r] = gws.ell[r];
  if (tid == 0) {
    if (ties && sh_ties) atomicAdd(ties, sh_ties);
    if (theta_out && T)
      *theta_out = n_star > 0 ? tau[n_star - 1] / T[R + n_star] : static_cast<double>(R) / T[R];
    if (K_out) *K_out = n_star;
  }
}

// ---------------------------------------------------------------------------
// Parallel path (up to kRankMaxN candidates): ranks over the whole GPU, then a
// one-CTA sweep in float-float arithmetic.
// ---------------------------------------------------------------------------
constexpr int kRankMaxN = 16384;   // candidates of the parallel path
constexpr int kRankThreads = 1024;
// keys of R runs at an odd stride: at most 8192 runs of 3 slots (gamma = 2)
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

  // this thread's keys in registers; the profile slice in shared memory (both
  // loaded once, up front, so that their latencies overlap)
  u64 kv[CHUNK];
#pragma unroll
  for (int q = 0; q < CHUNK; ++q) kv[q] = q < len ? gws.keysB[c0 + q] : 0ull;
  bool bad_t = false;
  if (T) {  // the top-K admission may run without a profile
    for (int m = tid; m <= n; m += blockDim.x) {
      const double t = T[R + m];
      const u64 b = static_cast<u64>(__double_as_longlong(t));
      if ((b >> 63) || ((b >> 52) & 0x7FFull) == 0x7FFull || b == 0ull) bad_t = true;
      sh_T[m] = t;
    }
  }
  if (bad_t) set_status(status, DSPARK_ERR_BAD_DATA);
  if (tid == 0) {
    sh_nE = 0;
    sh_break = INT_MAX;
    sh_ties = 0;
    sh_tau_star = ff{static_cast<float>(R), 0.f};
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
  ff tau_start = ff_add(ff{static_cast<float>(R), 0.f}, ex);
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
        const ff tau_m = ff_add(tau_prev, ff_from_bits(kv[q], okv));
        const double Tp = sh_T[m - 1], Tm = sh_T[m];
        const ff tm = ff_from_double(Tm, okv);
        bool improve, tie;
        if (okv) {
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
    Cand loc{0.0, 1.0, -1};
    ff tau_m = tau_start;
#pragma unroll
    for (int q = 0; q < CHUNK; ++q) {
      const int m = c0 + q + 1;
      if (q < len && m <= nE) {
        bool okv = true;
        tau_m = ff_add(tau_m, ff_from_bits(kv[q], okv));
        loc = cand_pick(loc, Cand{static_cast<double>(tau_m.hi) + tau_m.lo, sh_T[m], m});
      }
    }
    Cand run = cand_pick(Cand{static_cast<double>(R), sh_T[0], 0}, block_excl_pick(loc, sh_cand));
    unsigned n_ties = 0;
    tau_m = tau_start;
#pragma unroll
    for (int q = 0; q < CHUNK; ++q) {
      const int m = c0 + q + 1;
      if (q < len && m <= nE) {
        bool okv = true;
        tau_m = ff_add(tau_m, ff_from_bits(kv[q], okv));
        const Cand c{static_cast<double>(tau_m.hi) + tau_m.lo, sh_T[m], m};
        // |Theta(m) - Theta_best| <= eps Theta_best, multiplied through by both T
        if (fabs(c.tau * run.t - run.tau * c.t) <= DSPARK_SCHED_TIE_REL * run.tau * c.t) ++n_ties;
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
  for (int i = tid; i < n_star; i += blockDim.x) {
    const int id = gws.idxB[i];
    atomicMax(&sh_ell[id / gamma], id % gamma + 1);
  }
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
                              kSweepSmemMax) == cudaSuccess &&
         cudaFuncSetAttribute(k_sched_sweep<16, MODE>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSweepSmemMax) == cudaSuccess;
}

// the sweep instantiation whose per-thread chunk holds n / 1024 candidates
template <int MODE>
cudaError_t launch_sweep(int n, size_t smem, cudaStream_t st, const double* T, int R, int gamma,
                         const SchedWs& ws, int32_t* verify_len, double* theta, uint32_t* ties,
                         int32_t* status, const int32_t* K_in, int32_t* K_out) {
  if (n <= 4 * kRankThreads)
    return launch_pdl(k_sched_sweep<4, MODE>, 1, kRankThreads, smem, st, T, R, gamma, ws,
                      verify_len, theta, ties, status, K_in, K_out);
  if (n <= 8 * kRankThreads)
    return launch_pdl(k_sched_sweep<8, MODE>, 1, kRankThreads, smem, st, T, R, gamma, ws,
                      verify_len, theta, ties, status, K_in, K_out);
  return launch_pdl(k_sched_sweep<16, MODE>, 1, kRankThreads, smem, st, T, R, gamma, ws,
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
      if (cudaFuncSetAttribute(k_schedule, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSchedSmemMaxN * 24) != cudaSuccess)
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
    const int use_smem = n <= kSchedSmemMaxN ? 1 : 0;
    const size_t smem = use_smem ? static_cast<size_t>(n) * 24 : 0;
    if (launch_pdl(k_schedule, 1, kSchedThreads, smem, st, confidences, T, R, gamma, verify_len,
                   theta_best, ties, device_status, ws, use_smem, mode, K_in,
                   K_out) != cudaSuccess)
      return DSPARK_ERR_CUDA;
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
