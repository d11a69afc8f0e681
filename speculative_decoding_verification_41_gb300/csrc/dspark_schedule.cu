// dspark_schedule.cu -- hardware-aware prefix scheduler on GB300 (sm_103a).
//
// Method: "DSpark: Confidence-Scheduled Speculative Decoding with
// Semi-Autoregressive Generation", section 3.2.2, and Algorithm 1 of the
// Chinese translation page: prefix survival a_{r,j} = prod_{i<=j} c_{r,i}, a
// global descending sort of the candidates with a > 0, greedy admission along
// that order with Theta = tau * SPS(B) (SPS = 1/T), stop at the first
// Theta <= Theta_best.
//
// One CTA of 1024 threads:
//   1. survival products, one thread per request, multiplied left to right in
//      double (bit-identical to a sequential evaluation);
//   2. stable sort, descending: each request's run of gamma values is already
//      sorted (a is non-increasing in j), so runs are merged pairwise; every
//      element finds its output slot from its rank in the other run (binary
//      search), ties keep the flattened order. The keys are compared as the
//      64-bit patterns of the doubles, which order non-negative doubles exactly
//      (integer compares: GB300's double-precision rate is low). Keys and
//      indices live in shared memory up to 8192 candidates, in the workspace
//      beyond;
//   3. tau(n) = R + sum of the n largest a, as a block scan in double;
//   4. the first n with Theta(n) <= Theta(n-1) is found for every n in
//      parallel by a block min-reduction (every earlier step improved, so
//      Theta_best = Theta(n-1) there). Theta = tau / T is compared by
//      cross-multiplication, tau(n) T(R+n-1) vs tau(n-1) T(R+n), which decides
//      as the quotients do outside the 1e-9 near-tie window;
//   5. l_r = largest j among the first n* admitted candidates of request r.
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

__global__ void __launch_bounds__(kSchedThreads, 1)
    k_schedule(const float* __restrict__ conf, const double* __restrict__ T, int R, int gamma,
               int32_t* __restrict__ verify_len, double* theta_out, uint32_t* ties,
               int32_t* status, SchedWs gws, int use_smem) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ double red[32];
  __shared__ int red_i[32];
  __shared__ int sh_n_break, sh_nE;
  __shared__ unsigned sh_ties;
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
    *ties = 0;
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
  const int n_star = n_break <= nE ? n_break - 1 : nE;
  // near ties among the comparisons actually evaluated (steps 1..min(n_break, nE))
  {
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
  }
  // 5. verify lengths: the admitted prefix of each request
  for (int i = tid; i < n_star; i += kSchedThreads) {
    const int id = iA[i];
    atomicMax(&gws.ell[id / gamma], id % gamma + 1);
  }
  __syncthreads();
  for (int r = tid; r < R; r += kSchedThreads) verify_len[r] = gws.ell[r];
  if (tid == 0) {
    if (sh_ties) atomicAdd(ties, sh_ties);
    if (theta_out)
      *theta_out = n_star > 0 ? tau[n_star - 1] / T[R + n_star] : static_cast<double>(R) / T[R];
  }
}

std::mutex g_sched_mutex;
bool g_sched_ready[128];

}  // namespace dspark

extern "C" int dspark_schedule(const float* confidences, const double* step_time_ms,
                               int64_t n_profile, int32_t R, int32_t gamma, int32_t* verify_len,
                               double* theta_best, uint32_t* near_tie_count,
                               int32_t* device_status, void* workspace, size_t workspace_bytes,
                               struct CUstream_st* stream) {
  using namespace dspark;
  if (R < 1 || gamma < 1 || gamma > DSPARK_MAX_GAMMA) return DSPARK_ERR_INVALID_ARG;
  if (static_cast<long long>(R) * (gamma + 1) >= (1LL << 30)) return DSPARK_ERR_INVALID_ARG;
  if (!confidences || !step_time_ms || !verify_len || !device_status)
    return DSPARK_ERR_INVALID_ARG;
  if (n_profile < static_cast<int64_t>(R) * (gamma + 1) + 1) return DSPARK_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < DSPARK_SCHEDULE_WS_BYTES(R, gamma) ||
      reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return DSPARK_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return DSPARK_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(g_sched_mutex);
    if (!g_sched_ready[dev]) {
      if (cudaFuncSetAttribute(k_schedule, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSchedSmemMaxN * 24) != cudaSuccess)
        return DSPARK_ERR_CUDA;
      g_sched_ready[dev] = true;
    }
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
  const int use_smem = n <= kSchedSmemMaxN ? 1 : 0;
  const size_t smem = use_smem ? static_cast<size_t>(n) * 24 : 0;
  k_schedule<<<1, kSchedThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
      confidences, step_time_ms, R, gamma, verify_len, theta_best,
      near_tie_count ? near_tie_count : ws.ties_scratch, device_status, ws, use_smem);
  if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  return DSPARK_OK;
}
