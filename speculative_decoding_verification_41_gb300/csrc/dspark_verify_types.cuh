// dspark_verify_types.cuh -- constants, workspace records and compensated
// float helpers shared by the dspark_verify kernels (sm_103a).
#pragma once

#include <climits>

#include "dspark_common.cuh"

namespace dspark {

constexpr int kChunkBytes = 4096;               // one bulk copy
constexpr int kUnitBytes = DSPARK_TILE_BYTES;   // one work unit (one row statistic)
constexpr int kSeg = DSPARK_RESAMPLE_SEG;
static_assert(kUnitBytes % kChunkBytes == 0, "unit = whole chunks");

struct TileStat {  // statistics of one (row, unit): sum_v 2^(z_v*c - K) = s_hi + s_lo
  float s_hi;
  float s_lo;
  int32_t K;       // INT_MIN when the unit holds only masked (-inf) logits
  int32_t bad;     // non-zero if a non-finite maximum was met
};
static_assert(sizeof(TileStat) == 16, "TileStat layout");

struct ResampleDesc;  // the draw after a block (dspark_verify.cu)

struct WsHeader {
  int32_t total_rows;
  uint32_t ties_scratch;         // near-tie counter used when the caller passes none
  unsigned long long next_unit;  // claim counter of the streaming pass's last units
  unsigned long long next_item;  // claim counter of k_resid's last items (the draws)
  unsigned long long next_rate;  // claim counter of k_resid's last items (acceptance rates)
  int32_t pad[56];
};
static_assert(sizeof(WsHeader) == 256, "WsHeader layout");

struct VerifyWs {
  WsHeader* hdr;
  int32_t* req_row_start;  // [B+1]: first row-list entry of each request
  int64_t* row_list;       // [rows]: (global row << 1) | is_draft
  TileStat* tiles;         // [rows * n_units]
  ResampleDesc* desc;      // [B]
  ff* seg_sum;             // [B * n_seg]: per-segment weight sums as float pairs
  uint32_t* tickets;       // [B]
};

struct ExpParams {
  double c_d;  // log2(e) / T
  float c_hi;  // largest float <= c_d
  float c_lo;  // c_d - c_hi (> 0)
};

// ---------------------------------------------------------------------------
// compensated float helpers
// ---------------------------------------------------------------------------
// (hi, lo) <- (hi, lo) + (bh, bl), error-free transformation of the high parts
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float bh, float bl) {
  const float s = hi + bh;
  const float bp = s - hi;
  const float err = (hi - (s - bp)) + (bh - bp);
  hi = s;
  lo = lo + bl + err;
}

__device__ __forceinline__ void warp_two_sum(float& hi, float& lo) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xFFFFFFFFu, hi, o);
    const float ol = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
    two_sum_acc(hi, lo, oh, ol);
  }
}

// x * 2^d for d <= 0 (exact while the result stays normal)
__device__ __forceinline__ float scale_pow2(float x, int d) { return d < -200 ? 0.f : ldexpf(x, d); }

// 2^(z*c - K), with z*c formed from c_hi + c_lo so that the rounding of c does
// not bias the sum; -inf logits give 0.
__device__ __forceinline__ float exp_term(float z, float nK, const ExpParams& ep) {
  return ex2_approx(fmaf(z, ep.c_lo, fmaf(z, ep.c_hi, nK)));
}

}  // namespace dspark
