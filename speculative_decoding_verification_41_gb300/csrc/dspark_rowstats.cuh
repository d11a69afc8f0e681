// dspark_rowstats.cuh -- the streaming pass of dspark_verify: per-unit
// softmax statistics of every needed logit row (sm_103a).
#pragma once

#include "dspark_verify_types.cuh"

namespace dspark {

// ---------------------------------------------------------------------------
// k_rowstats: unit statistics
// ---------------------------------------------------------------------------
// Per-lane running state of one unit.
struct LaneAcc {
  int32_t K = INT_MIN;  // exponent reference (INT_MIN: nothing seen yet)
  float s = 0.f;        // Kahan sum of 2^(z*c - K)
  float comp = 0.f;     // Kahan compensation (value = s - comp)
  bool bad = false;
};

// Raise the lane's reference if a chunk maximum outgrows it by more than 2^64
// (first chunk: set it). Returns -K as float for the FMA chain.
__device__ __forceinline__ float lane_reference(LaneAcc& a, float lane_max, const ExpParams& ep) {
  if (lane_max > -INFINITY) {
    const float mc = lane_max * ep.c_hi;
    if (!(fabsf(mc) < 1.0e9f)) {  // +inf / NaN / absurd logits
      a.bad = true;
    } else if (a.K == INT_MIN || mc > static_cast<float>(a.K) + 64.f) {
      const int Kn = static_cast<int>(ceilf(mc));
      if (a.K != INT_MIN) {
        a.s = scale_pow2(a.s, a.K - Kn);
        a.comp = scale_pow2(a.comp, a.K - Kn);
      }
      a.K = Kn;
    }
  }
  return a.K == INT_MIN ? 0.f : -static_cast<float>(a.K);
}

__device__ __forceinline__ void kahan_add(LaneAcc& a, float x) {
  const float y = x - a.comp;
  const float t = a.s + y;
  a.comp = (t - a.s) - y;
  a.s = t;
}

// One 4 KB chunk held in registers (VPL 16-byte vectors per lane).
template <typename Tin, int VPL>
__device__ __forceinline__ void chunk_accumulate(const uint4 (&v)[VPL], LaneAcc& a,
                                                 const ExpParams& ep) {
  float lane_max;
  if constexpr (sizeof(Tin) == 2) {
    __nv_bfloat162 m2 = *reinterpret_cast<const __nv_bfloat162*>(&v[0].x);
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v[j]);
      m2 = __hmax2(m2, __hmax2(__hmax2(p[0], p[1]), __hmax2(p[2], p[3])));
    }
    lane_max = fmaxf(__low2float(m2), __high2float(m2));
  } else {
    lane_max = -INFINITY;
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      lane_max = fmaxf(lane_max, fmaxf(fmaxf(__uint_as_float(v[j].x), __uint_as_float(v[j].y)),
                                       fmaxf(__uint_as_float(v[j].z), __uint_as_float(v[j].w))));
  }
  if (!(lane_max > -INFINITY)) {
    if (lane_max != lane_max) a.bad = true;  // NaN
    return;
  }
  const float nK = lane_reference(a, lane_max, ep);
  float part[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    if constexpr (sizeof(Tin) == 2) {
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
      float e[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        e[2 * q] = exp_term(bf16_lo(w[q]), nK, ep);
        e[2 * q + 1] = exp_term(bf16_hi(w[q]), nK, ep);
      }
      part[j] = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
    } else {
      const float e0 = exp_term(__uint_as_float(v[j].x), nK, ep);
      const float e1 = exp_term(__uint_as_float(v[j].y), nK, ep);
      const float e2 = exp_term(__uint_as_float(v[j].z), nK, ep);
      const float e3 = exp_term(__uint_as_float(v[j].w), nK, ep);
      part[j] = (e0 + e1) + (e2 + e3);
    }
  }
#pragma unroll
  for (int w = 1; w < VPL; w <<= 1)
#pragma unroll
    for (int j = 0; j + w < VPL; j += 2 * w) part[j] += part[j + w];
  kahan_add(a, part[0]);
}

// End of a unit: merge the lanes (exact power-of-two alignment, TwoSum) and
// write the statistics.
__device__ __forceinline__ void unit_finish(const LaneAcc& a, TileStat* out, int lane,
                                            int32_t* status) {
  const int Kw = __reduce_max_sync(0xFFFFFFFFu, a.K);
  const bool bad = __any_sync(0xFFFFFFFFu, a.bad);
  float hi = 0.f, lo = 0.f;
  if (a.K != INT_MIN) {
    hi = scale_pow2(a.s, a.K - Kw);
    lo = -scale_pow2(a.comp, a.K - Kw);
  }
  warp_two_sum(hi, lo);
  if (lane == 0) {
    TileStat ts;
    const float s = hi + lo;  // renormalise the pair
    ts.s_hi = s;
    ts.s_lo = lo - (s - hi);
    ts.K = Kw;
    ts.bad = bad ? 1 : 0;
    if (bad) set_status(status, DSPARK_ERR_BAD_DATA);
    *out = ts;
  }
}

// Streaming pass through the TMA engine. Row byte length and both buffers
// must be 16-byte aligned. Shared memory: W warps x STAGES x (4 KB + barrier +
// 16-byte chunk record).
//
// Work assignment: warp gw takes units gw, gw + GW, ... among the first
// U - U/kDynamicDiv units, then claims the remaining ones (about
// 1/kDynamicDiv) one at a time from a counter (reset by k_plan). A CTA that starts late
// -- its SM still held by another kernel, e.g. a scheduler running on another
// stream -- then takes fewer of the last units instead of finishing late. The
// producer (lane 0) records which unit and bytes each stage holds, so the
// consumer follows whatever the claims gave.
constexpr int kDynamicDiv = 8;

struct __align__(16) ChunkRec {  // what a ring stage holds; written by lane 0
  long long u;    // unit (row-list row * n_units + part)
  int32_t bytes;  // bytes of the chunk
  int32_t last;   // the unit's last chunk
};
static_assert(sizeof(ChunkRec) == 16, "ChunkRec layout");

template <typename Tin, int W, int STAGES>
__global__ void __launch_bounds__(W * 32, 1)
    k_rowstats_tma(const Tin* __restrict__ tl, const Tin* __restrict__ dl, int V, int n_units,
                   VerifyWs ws, ExpParams ep, int32_t* status) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  constexpr int VPL = kChunkBytes / 16 / 32;  // 16-byte vectors per lane per chunk
  extern __shared__ __align__(1024) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* buf = smem + static_cast<size_t>(warp) * STAGES * kChunkBytes;
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(W) * STAGES * kChunkBytes) +
      warp * STAGES;
  ChunkRec* recs =
      reinterpret_cast<ChunkRec*>(smem + static_cast<size_t>(W) * STAGES * (kChunkBytes + 8)) +
      warp * STAGES;
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  const long long U = static_cast<long long>(ws.hdr->total_rows) * n_units;
  const long long gw = static_cast<long long>(blockIdx.x) * W + warp;
  const long long GW = static_cast<long long>(gridDim.x) * W;
  const long long row_bytes = static_cast<long long>(V) * sizeof(Tin);
  // the first S units in fixed rounds (warp gw: gw, gw + GW, ... below S),
  // the last U - S (about 1/kDynamicDiv) claimed
  const long long S = U - U / kDynamicDiv;
  const long long n_static = gw < S ? (S - 1 - gw) / GW + 1 : 0;
  const long long dyn0 = S;  // first unit of the claims

  // producer cursor (lane 0): the unit being copied and its next chunk
  long long k_st = 0;
  auto next_unit = [&]() -> long long {
    if (k_st < n_static) return gw + (k_st++) * GW;
    return dyn0 + static_cast<long long>(atomicAdd(&ws.hdr->next_unit, 1ull));
  };
  long long pu = 0;
  int pc = 0, pub = 0;
  bool have = false;
  const char* pbase = nullptr;
  auto issue_next = [&](int s) {  // lane 0 only; have
    if (pc == 0) {
      const long long row = pu / n_units;
      const long long part = pu - row * n_units;
      const long long e = ws.row_list[row];
      pbase = reinterpret_cast<const char*>((e & 1) ? dl : tl) + (e >> 1) * row_bytes +
              part * static_cast<long long>(kUnitBytes);
      const long long left = row_bytes - part * kUnitBytes;
      pub = static_cast<int>(left < kUnitBytes ? left : kUnitBytes);
    }
    const int left = pub - pc * kChunkBytes;
    const uint32_t bytes = static_cast<uint32_t>(left < kChunkBytes ? left : kChunkBytes);
    ChunkRec rc;
    rc.u = pu;
    rc.bytes = static_cast<int>(bytes);
    rc.last = left <= kChunkBytes;
    recs[s] = rc;
    mbar_arrive_expect_tx(&bars[s], bytes);
    bulk_g2s(buf + s * kChunkBytes, pbase + static_cast<long long>(pc) * kChunkBytes, bytes,
             &bars[s]);
    if (rc.last) {
      pc = 0;
      pu = next_unit();
      have = pu < U;
    } else {
      ++pc;
    }
  };
  int inflight = 0;
  if (lane == 0) {
    pu = next_unit();
    have = pu < U;
    while (inflight < STAGES && have) issue_next(inflight++);
  }
  inflight = __shfl_sync(0xFFFFFFFFu, inflight, 0);

  int stage = 0;
  uint32_t phase = 0;
  uint4 neg_inf;
  neg_inf.x = neg_inf.y = neg_inf.z = neg_inf.w = (sizeof(Tin) == 2) ? 0xFF80FF80u : 0xFF800000u;
  LaneAcc acc;
  while (inflight > 0) {
    // every lane waits (each gets the barrier's acquire); the give-up decision is warp-uniform
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bars[stage], phase))) {
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
    const ChunkRec rc = recs[stage];
    uint4 v[VPL];
    const uint4* sp = reinterpret_cast<const uint4*>(buf + stage * kChunkBytes);
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int idx = j * 32 + lane;
      v[j] = (idx * 16 < rc.bytes) ? sp[idx] : neg_inf;
    }
    __syncwarp();
    const int freed = stage;
    if (++stage == STAGES) {
      stage = 0;
      phase ^= 1u;
    }
    --inflight;
    if (lane == 0 && have) {  // the ring was full: the freed stage is the next one to fill
      fence_proxy_async();
      issue_next(freed);
      ++inflight;
    }
    inflight = __shfl_sync(0xFFFFFFFFu, inflight, 0);
    chunk_accumulate<Tin, VPL>(v, acc, ep);
    if (rc.last) {
      unit_finish(acc, ws.tiles + rc.u, lane, status);
      acc = LaneAcc();
    }
  }
}

// Fallback streaming pass with plain loads, for rows whose byte length or
// buffers are not 16-byte aligned.
template <typename Tin>
__global__ void __launch_bounds__(256) k_rowstats_plain(const Tin* __restrict__ tl,
                                                        const Tin* __restrict__ dl, int V,
                                                        int n_units, VerifyWs ws, ExpParams ep,
                                                        int32_t* status) {
  pdl_wait();  // predecessor grid complete, its writes visible
  pdl_trigger();
  constexpr int kUnitElems = kUnitBytes / sizeof(Tin);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long U = static_cast<long long>(ws.hdr->total_rows) * n_units;
  const long long GW = static_cast<long long>(gridDim.x) * 8;
  for (long long u = static_cast<long long>(blockIdx.x) * 8 + warp; u < U; u += GW) {
    const long long row = u / n_units;
    const int part = static_cast<int>(u - row * n_units);
    const long long e = ws.row_list[row];
    const Tin* src = ((e & 1) ? dl : tl) + (e >> 1) * static_cast<long long>(V) +
                     static_cast<long long>(part) * kUnitElems;
    const int n = min(kUnitElems, V - part * kUnitElems);
    float mx = -INFINITY;
    for (int i = lane; i < n; i += 32) mx = fmaxf(mx, to_float<Tin>(src[i]));
    LaneAcc acc;
    const float nK = lane_reference(acc, mx, ep);
    if (mx != mx) acc.bad = true;
    if (acc.K != INT_MIN) {
      for (int i = lane; i < n; i += 32) kahan_add(acc, exp_term(to_float<Tin>(src[i]), nK, ep));
    }
    unit_finish(acc, ws.tiles + u, lane, status);
  }
}

}  // namespace dspark
