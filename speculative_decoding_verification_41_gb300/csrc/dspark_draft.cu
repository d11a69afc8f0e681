// dspark_draft.cu -- the sequential stage of the DSpark drafter with the
// Markov head, on one GB300 (sm_103a).
//
// DSpark paper, section 3.1 ("Sequential stage"): the block is drawn left to
// right from p_k(v) = softmax(U_k + B_k)(v) (equation 4), with the Markov head's
// transition bias B(x_{k-1}, .) = W1[x_{k-1}] W2 (equation 5, W1 of V x r, W2 of
// r x V, r = 256 by default). Every position is one pass of two kernels:
//
//   k_draft_step  (tensor cores) D = G W2 for the batch, G[b] = W1[x_{k-1}(b)]:
//                 an M = requests x N = vocabulary x K = r product by
//                 tcgen05.mma (bf16 in, f32 accumulators in tensor memory).
//                 G stays in tensor memory for the whole launch (the MMA's
//                 A operand), so shared memory holds only the W2 stream,
//                 brought in by tiled TMA in the 128-byte swizzled layout,
//                 and the U / L tiles. The epilogue adds U_k, rounds to bf16 (the emitted
//                 draft row that the verifier reads), stores it by TMA and
//                 writes one softmax statistic per (request, 128-token tile).
//   k_draft_pick  (one warp per request) merges the tile statistics, finds the
//                 tile where the running sum crosses u*Z, re-reads that tile's
//                 128 emitted logits and returns the token: an inverse-CDF
//                 draw of softmax(L_k / T) in ascending token order. It then
//                 copies W1[x_k] into G for the next position.
//
// dspark_draft_markov runs the whole block in one cooperative launch where the
// grid fits on the GPU at once: k_draft_pair for two request tiles
// (128 < B <= 256: the streaming CTAs serve both tiles and the draws run on
// CTAs of their own, so one tile's draws and next G overlap the other tile's
// streaming), k_draft_block otherwise (the CTAs of a request tile stream it,
// meet at a barrier, draw); larger grids, and the timed entry point, take the
// two kernels per position above.
//
// W2 is stored transposed, w2t[v][j] = W2[j][v], so both operands are K-major.
// The tile is 128 requests x 128 tokens. With G in tensor memory (where the
// MMA reads it without touching shared memory), a ring of 8 W2 chunks keeps two
// tiles of rank 256 in flight beside 3 U / L slots, so the W2 stream is not
// serialised on one memory latency per tile, and each MMA reads only its 4 KB
// W2 slice from shared memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "dspark_sync.cuh"
#include "dspark_tc.cuh"
#include "dspark_verify_types.cuh"

namespace dspark {
namespace {

constexpr int kDM = 128;                             // requests per tile (MMA M)
constexpr int kDN = DSPARK_DRAFT_TILE;               // vocabulary per tile (MMA N)
constexpr int kDK = 64;                              // K per chunk: one 128-byte row of bf16
constexpr int kDStages = 8;  // W2 ring: 128 x 64 chunks, two tiles of rank 256 in flight
constexpr int kDSlots = 3;   // U / L tile slots
constexpr int kDEpiWarps = 8;                        // two groups of four (warps 2..9)
constexpr int kDThreads = 96 + kDEpiWarps * 32;      // W2 producer, MMA, epilogue, U producer
constexpr int kDWarpU = 2 + kDEpiWarps;              // the U producer's warp
constexpr uint32_t kBoxW = kDN * 128u;               // W2 chunk: 128 vocabulary rows x 128 B
constexpr uint32_t kBoxU = kDM * 128u;               // half a U / L tile: 128 rows x 64 bf16
constexpr uint32_t kOffW = 0;
constexpr uint32_t kOffU = kOffW + kDStages * kBoxW;
constexpr uint32_t kOffBar = kOffU + kDSlots * 2 * kBoxU;
constexpr uint32_t kDraftSmem = kOffBar + 512 + 1024;  // barriers, 1024-byte alignment slack
// Tensor memory: two f32 accumulators of kDN columns, then G = W1[x_{k-1}] of
// the request tile (row m in lane m, two bf16 per column: r / 2 columns).
constexpr uint32_t kColG = 2 * kDN;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = idesc_bf16_f32(kDM, kDN);
static_assert(kDN == 128 && kDK == 64, "epilogue and statistics assume 128-token tiles");
static_assert(kColG + DSPARK_DRAFT_MAX_RANK / 2 <= kTmemCols, "tensor memory columns");

// A request's token flag sits alone on a 128-byte line (16 words): every
// streaming CTA polls the flags, and packed 16 to a line their reads all land
// on a few L2 slices, which cost the block up to a fifth of its time
// depending on where the workspace happened to start.
constexpr int kReadyStride = 16;

static_assert(kDraftSmem <= 232448, "shared memory of k_draft_step");
// more than half of an SM's 228 KB: one CTA per SM (the single launch maps CTAs by SM id)
static_assert(kDraftSmem > 233472 / 2, "one drafter CTA per SM");

struct DraftStat {  // one (request, tile): sum over the tile of 2^(L_v * c - R)
  float s;
  int32_t R;  // INT_MIN when every logit of the tile is -inf
};

struct DraftBars {
  uint64_t a_full;  // G is in tensor memory (one arrival per epilogue warp)
  uint64_t w_full[kDStages], w_empty[kDStages];
  uint64_t u_full[kDSlots], u_empty[kDSlots];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t st_ready[2];  // a group's rows are in shared memory, ready to store
  uint64_t mma_done;
  uint64_t epi_done;     // k_draft_block: the CTA's epilogue warps reached the tile barrier
  uint64_t step_go;      // k_draft_block: the tile barrier was crossed
  uint32_t tmem_base;
};
static_assert(sizeof(DraftBars) <= 512, "barrier block");

struct DraftStepArgs {
  int32_t B, V, r, gamma, k;
  int32_t n_tiles;  // vocabulary tiles
  int32_t n_m;      // request tiles
  int32_t per_m;    // CTAs per request tile
  ExpParams ep;
  DraftStat* stats;  // [B][n_tiles]
  int32_t* status;
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
// two floats -> packed bf16x2 (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Wait with a bound; on timeout record DSPARK_ERR_TIMEOUT and report failure.
__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_wait(bar, parity)) return true;
  set_status(status, DSPARK_ERR_TIMEOUT);
  return false;
}

// Exponent reference of a chunk whose largest logit is cm: R = ceil(cm * c_hi)
// (INT_MIN for an all -inf chunk). The draw recomputes it the same way.
__device__ __forceinline__ int32_t chunk_reference(float cm, float c_hi) {
  return cm > -INFINITY && cm < INFINITY ? static_cast<int32_t>(ceilf(cm * c_hi)) : INT_MIN;
}

// One epilogue tile of one thread: its request row m, 128 columns from
// tensor memory (taddr) and from the U slot (ubase: two boxes of 64 columns,
// 128-byte swizzled rows). Writes the rounded row over U. Each 32-column chunk
// c gets its own reference R_c and the pairwise sum S_c of 2^(L*c - R_c); the
// tile statistic is (R, S) with R = max R_c and S = sum_c S_c 2^(R_c - R), the
// chunks folded in order by exact power-of-two scaling. FULL: every column is
// inside the vocabulary (no masks). Releases the accumulator (acc_empty) once
// its last columns are in registers.
template <bool FULL>
__device__ __forceinline__ void epi_tile(uint32_t taddr, uint32_t ubase, int m, int v0, int V,
                                         const ExpParams& ep, int32_t& R_out, float& S_out,
                                         bool& inf_seen, uint64_t* acc_empty, int lane) {
  int32_t Rt = INT_MIN;
  float St = 0.f;
#pragma unroll 1
  for (int c4 = 0; c4 < 4; ++c4) {
    float acc[32];
    __syncwarp();
    tmem_ld32(taddr + c4 * 32, acc);
    if (c4 == 3) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
    }
    const uint32_t row = ubase + (c4 >> 1) * kBoxU + m * 128;
    uint32_t lw[16];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const uint32_t addr = row + (((((c4 & 1) * 4) + jj) ^ (m & 7)) << 4);
      const uint4 u = lds128(addr);
      lw[4 * jj + 0] = pack_bf16x2(acc[8 * jj + 0] + bf16_lo(u.x), acc[8 * jj + 1] + bf16_hi(u.x));
      lw[4 * jj + 1] = pack_bf16x2(acc[8 * jj + 2] + bf16_lo(u.y), acc[8 * jj + 3] + bf16_hi(u.y));
      lw[4 * jj + 2] = pack_bf16x2(acc[8 * jj + 4] + bf16_lo(u.z), acc[8 * jj + 5] + bf16_hi(u.z));
      lw[4 * jj + 3] = pack_bf16x2(acc[8 * jj + 6] + bf16_lo(u.w), acc[8 * jj + 7] + bf16_hi(u.w));
      sts128(addr, make_uint4(lw[4 * jj], lw[4 * jj + 1], lw[4 * jj + 2], lw[4 * jj + 3]));
    }
    const int vc = v0 + c4 * 32;  // first column of the chunk
    float cm;
    if constexpr (FULL) {
      __nv_bfloat162 h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        h[i] = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&lw[2 * i]),
                       *reinterpret_cast<const __nv_bfloat162*>(&lw[2 * i + 1]));
#pragma unroll
      for (int w = 4; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) h[i] = __hmax2(h[i], h[i + w]);
      cm = fmaxf(__low2float(h[0]), __high2float(h[0]));
    } else {
      cm = -INFINITY;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (vc + 2 * i < V) cm = fmaxf(cm, bf16_lo(lw[i]));
        if (vc + 2 * i + 1 < V) cm = fmaxf(cm, bf16_hi(lw[i]));
      }
    }
    inf_seen |= !(cm < INFINITY) && !(cm == -INFINITY);  // +inf or NaN
    const int32_t R = chunk_reference(cm, ep.c_hi);
    float e[32];
    const float nK = R == INT_MIN ? 0.f : -static_cast<float>(R);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      e[2 * i] = exp_term(bf16_lo(lw[i]), nK, ep);
      e[2 * i + 1] = exp_term(bf16_hi(lw[i]), nK, ep);
      if constexpr (!FULL) {
        if (vc + 2 * i >= V) e[2 * i] = 0.f;
        if (vc + 2 * i + 1 >= V) e[2 * i + 1] = 0.f;
      }
    }
#pragma unroll
    for (int w = 16; w > 0; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) e[i] += e[i + w];
    if (R != INT_MIN) {
      if (R > Rt) {
        St = Rt == INT_MIN ? 0.f : scale_pow2(St, Rt - R);
        Rt = R;
        St += e[0];
      } else {
        St += scale_pow2(e[0], R - Rt);
      }
    }
  }
  R_out = Rt;
  S_out = St;
}

// ---------------------------------------------------------------------------
// k_draft_gather: G[b] = W1[x_0(b)] before the first position
// ---------------------------------------------------------------------------
__device__ __forceinline__ void copy_row(const uint16_t* __restrict__ W1, uint16_t* __restrict__ G,
                                         int x, int b, int r, int lane) {
  const uint4* src = reinterpret_cast<const uint4*>(W1 + static_cast<size_t>(x) * r);
  uint4* dst = reinterpret_cast<uint4*>(G + static_cast<size_t>(b) * r);
  for (int i = lane; i < r / 8; i += 32) dst[i] = src[i];
}

__global__ void __launch_bounds__(32) k_draft_gather(const int32_t* __restrict__ anchors,
                                                     const uint16_t* __restrict__ W1,
                                                     uint16_t* __restrict__ G, int B, int V, int r,
                                                     int32_t* status) {
  const int b = blockIdx.x;
  if (b >= B) return;
  int x = anchors[b];
  if (x < 0 || x >= V) {
    if (threadIdx.x == 0) set_status(status, DSPARK_ERR_BAD_DATA);
    x = 0;
  }
  copy_row(W1, G, x, b, r, threadIdx.x);
}

// ---------------------------------------------------------------------------
// k_draft_pick: inverse-CDF draw of position k for one request
// ---------------------------------------------------------------------------
struct DraftPickArgs {
  int32_t B, V, r, gamma, k, n_tiles;
  ExpParams ep;
  const DraftStat* stats;    // [B][n_tiles]
  const uint16_t* L;         // emitted rows [B][gamma][V]
  const float* uniforms;     // [B][gamma]
  const uint16_t* W1;        // [V][r]
  uint16_t* G;               // [B][r]
  int32_t* tokens;           // [B][gamma]
  int32_t* status;
  unsigned long long* ready;  // k_draft_block: [B], (k + 1) << 32 | x_k once drawn
  bool relaxed_flag = false;  // the flag's reader needs only x_k (k_draft_pair)
};

constexpr int kPickWarps = 4;   // one request per warp
constexpr int kPickBatch = 32;  // statistics loaded per round trip by a lane

// A statistic through the read-only path (kCoherent false: written by an
// earlier kernel) or through L2 only (written earlier in this kernel, at an
// address reused every position).
template <bool kCoherent>
__device__ __forceinline__ DraftStat ld_stat(const DraftStat* p) {
  int2 v;
  if constexpr (kCoherent)
    asm volatile("ld.global.cg.v2.s32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  else
    v = __ldg(reinterpret_cast<const int2*>(p));
  return DraftStat{__int_as_float(v.x), v.y};
}
template <bool kCoherent>
__device__ __forceinline__ uint2 ld_u2(const uint16_t* p) {
  uint2 v;
  if constexpr (kCoherent)
    asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  else
    v = *reinterpret_cast<const uint2*>(p);
  return v;
}

// 2^d for d <= 0 as a float, built from its exponent bits (0 below the
// normal range, where a term is far below any mass that can decide a draw).
__device__ __forceinline__ float pow2_nonpos(int d) {
  return d < -126 ? 0.f : __int_as_float((d + 127) << 23);
}

__device__ __forceinline__ ff ff_scale(ff v, float p2) { return ff{v.hi * p2, v.lo * p2}; }

__device__ __forceinline__ ff warp_incl_scan_ff(ff v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff u = shfl_up_ff(v, o);
    if (lane >= o) v = ff_add(v, u);
  }
  return v;
}

// The token inside crossing tile g of request b: the tile's 128 terms
// recomputed exactly as the tile kernel did (each 32-column chunk (8 lanes)
// with its own reference, scaled to the request's Rmax), scanned on from
// s_before to the first running sum above target. All lanes of one warp.
template <bool kCoherent>
__device__ __forceinline__ int draw_in_tile(const DraftPickArgs& a, int b, int g, ff s_before,
                                            ff target, int32_t Rmax, int lane) {
  // the crossing tile: recompute its 128 terms exactly as the step kernel
  // did, each 32-column chunk (8 lanes) with its own reference
  const int v = g * kDN + 4 * lane;
  float z[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  if (v < a.V) {  // V is a multiple of 8: v + 3 < V too
    const uint2 raw =
        ld_u2<kCoherent>(a.L + (static_cast<size_t>(b) * a.gamma + a.k) * a.V + v);
    z[0] = bf16_lo(raw.x);
    z[1] = bf16_hi(raw.x);
    z[2] = bf16_lo(raw.y);
    z[3] = bf16_hi(raw.y);
  }
  float cm = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, o));
  const int32_t Rc = chunk_reference(cm, a.ep.c_hi);
  float w[4] = {0.f, 0.f, 0.f, 0.f};
  if (Rc != INT_MIN && v < a.V) {
    const float nK = -static_cast<float>(Rc);
    const float scale = pow2_nonpos(Rc - Rmax);
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = exp_term(z[e], nK, a.ep) * scale;
  }
  ff lsum{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 4; ++e) lsum = ff_add(lsum, ff{w[e], 0.f});
  const ff inc_l = warp_incl_scan_ff(lsum, lane);
  const ff pre = shfl_up_ff(inc_l, 1);
  const ff base = ff_add(s_before, lane > 0 ? pre : ff{0.f, 0.f});
  const uint32_t cross = __ballot_sync(0xFFFFFFFFu, ff_cmp(ff_add(s_before, inc_l), target) > 0);
  int pick = -1;
  if (cross) {
    const int L0 = __ffs(cross) - 1;
    if (lane == L0) {
      ff c = base;
      int last = -1;
      for (int e = 0; e < 4; ++e) {
        if (w[e] > 0.f) last = e;
        const ff nc = ff_add(c, ff{w[e], 0.f});
        if (w[e] > 0.f && ff_cmp(nc, target) > 0) {
          pick = v + e;
          break;
        }
        c = nc;
      }
      if (pick < 0) pick = v + (last >= 0 ? last : 0);
    }
    pick = __shfl_sync(0xFFFFFFFFu, pick, L0);
  } else {  // rounding: the last token of the tile with positive weight
    const int lpos = (w[3] > 0.f) ? 3 : (w[2] > 0.f) ? 2 : (w[1] > 0.f) ? 1 : (w[0] > 0.f) ? 0 : -1;
    const uint32_t any = __ballot_sync(0xFFFFFFFFu, lpos >= 0);
    const int Lh = any ? 31 - __clz(any) : 0;
    const int e = __shfl_sync(0xFFFFFFFFu, lpos, Lh);
    pick = g * kDN + 4 * Lh + (e >= 0 ? e : 0);
  }
  return pick;
}

// The drawn token out: the tokens array, then either the ready flag the single
// launch's next position waits on (with W1[x_k] pulled into L2 first, so that
// the CTAs loading it hit L2) or the row G[b] = W1[x_k] the next launch reads.
__device__ __forceinline__ void publish_token(const DraftPickArgs& a, int b, int y, int lane) {
  if (lane == 0) a.tokens[static_cast<size_t>(b) * a.gamma + a.k] = y;
  if (a.ready) {
    if (a.k + 1 < a.gamma && lane * 128 < a.r * 2) {
      const char* line = reinterpret_cast<const char*>(a.W1 + static_cast<size_t>(y) * a.r) +
                         lane * 128;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
    }
    if (lane == 0 && a.k + 1 < a.gamma) {
      const unsigned long long f =
          (static_cast<unsigned long long>(a.k + 1) << 32) | static_cast<uint32_t>(y);
      // k_draft_pair's reader takes only the token from the flag (W1 is an
      // input): no ordering needed; k_draft_block's readers rely on a release
      if (a.relaxed_flag)
        asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(&a.ready[b * kReadyStride]), "l"(f) : "memory");
      else
        st_release_gpu64(&a.ready[b * kReadyStride], f);
    }
  } else if (a.k + 1 < a.gamma) {
    copy_row(a.W1, a.G, y, b, a.r, lane);
  }
}

// One warp draws position k of request b from the tile statistics of an
// earlier kernel, in float-float arithmetic (about 48 significant bits; this
// GPU's FP64 rate is far too low for it): the lanes own contiguous runs of
// the request's tile statistics, a scan gives every lane its exclusive prefix
// (the next lane's exclusive prefix is bitwise this lane's inclusive one, so
// the lanes partition [0, Z)), the owning lane walks its run to the crossing
// tile, and draw_in_tile recomputes that tile's 128 terms exactly as the step
// kernel did and draws.
template <bool kCoherent>
__device__ __forceinline__ void draw_request(const DraftPickArgs& a, int b, int lane) {
  const DraftStat* st = a.stats + static_cast<size_t>(b) * a.n_tiles;
  const int per = (a.n_tiles + 31) / 32;
  const int g0 = lane * per < a.n_tiles ? lane * per : a.n_tiles;
  const int g1 = g0 + per < a.n_tiles ? g0 + per : a.n_tiles;

  // one pass over the lane's tiles, loads issued kPickBatch at a time (all at
  // once, and kept for the walk below, when they fit): the lane's largest
  // reference Rl and its mass Sl = sum s 2^(R - Rl), rescaled exactly whenever
  // Rl grows
  int32_t Rl = INT_MIN;
  ff Sl{0.f, 0.f};
  DraftStat d[kPickBatch];
  const bool held = per <= kPickBatch;
  for (int gb = g0; gb < g1; gb += kPickBatch) {
#pragma unroll
    for (int i = 0; i < kPickBatch; ++i)
      d[i] = gb + i < g1 ? ld_stat<kCoherent>(st + gb + i) : DraftStat{0.f, INT_MIN};
#pragma unroll
    for (int i = 0; i < kPickBatch; ++i) {
      if (!(d[i].s > 0.f)) continue;
      if (d[i].R > Rl) {
        Sl = Rl == INT_MIN ? ff{0.f, 0.f} : ff_scale(Sl, pow2_nonpos(Rl - d[i].R));
        Rl = d[i].R;
      }
      Sl = ff_add(Sl, ff{d[i].s * pow2_nonpos(d[i].R - Rl), 0.f});
    }
  }
  int32_t Rmax = Rl;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Rmax = max(Rmax, __shfl_xor_sync(0xFFFFFFFFu, Rmax, o));
  const float u = a.uniforms[static_cast<size_t>(b) * a.gamma + a.k];
  int y = 0;
  if (Rmax == INT_MIN || !(u >= 0.f && u < 1.f)) {
    if (lane == 0) set_status(a.status, DSPARK_ERR_BAD_DATA);
  } else {
    const ff S = Rl == INT_MIN ? ff{0.f, 0.f} : ff_scale(Sl, pow2_nonpos(Rl - Rmax));
    const bool has = S.hi > 0.f;
    const ff incl = warp_incl_scan_ff(S, lane);
    const ff Z = shfl_ff(incl, 31);
    const ff prev = shfl_up_ff(incl, 1);
    const ff excl = lane > 0 ? prev : ff{0.f, 0.f};
    const ff target = ff_mul(ff{u, 0.f}, Z);
    const uint32_t own =
        __ballot_sync(0xFFFFFFFFu, has && ff_cmp(excl, target) <= 0 && ff_cmp(target, incl) < 0);
    int gs = -1;
    ff before{0.f, 0.f};
    if (own && lane == __ffs(own) - 1) {  // walk this lane's tiles (in registers when they fit)
      ff C = excl, Clast = excl;
      int glast = -1;
      for (int gb = g0; gb < g1 && gs < 0; gb += kPickBatch) {
        if (!held) {
#pragma unroll
          for (int i = 0; i < kPickBatch; ++i)
            d[i] = gb + i < g1 ? ld_stat<kCoherent>(st + gb + i) : DraftStat{0.f, INT_MIN};
        }
#pragma unroll
        for (int i = 0; i < kPickBatch; ++i) {
          if (gs >= 0 || !(d[i].s > 0.f)) continue;
          const ff next = ff_add(C, ff{d[i].s * pow2_nonpos(d[i].R - Rmax), 0.f});
          if (ff_cmp(next, target) > 0) {
            gs = gb + i;
          } else {
            glast = gb + i;
            Clast = C;
            C = next;
          }
        }
      }
      if (gs < 0) {  // rounding left the target past this lane's last tile: take it
        gs = glast;
        C = Clast;
      }
      before = C;
    }
    const int ol = own ? __ffs(own) - 1 : 0;
    const int g = own ? __shfl_sync(0xFFFFFFFFu, gs, ol) : -1;
    const ff s_before = shfl_ff(before, ol);
    if (g >= 0) y = draw_in_tile<kCoherent>(a, b, g, s_before, target, Rmax, lane);
  }
  publish_token(a, b, y, lane);
}

// The vocabulary tiles of a request tile are split into per_m contiguous
// ranges, one per CTA: range p is [range_begin(p), range_begin(p + 1)).
__device__ __forceinline__ int range_begin(int p, int n_tiles, int per_m) {
  return static_cast<int>(static_cast<long long>(p) * n_tiles / per_m);
}

// One request's softmax mass over one CTA's range of tiles at one position:
// sum 2^(L_v * c - R) = hi + lo (a float pair), R the largest tile reference
// of the range (INT_MIN if every term is 0). The single launch's draws scan
// these first, then the tiles of the one range holding the cut.
struct __align__(16) DraftPartial {
  float hi, lo;
  int32_t R;
  int32_t pad;
};
// Partial records the workspace holds per position parity: per_m ranges of
// 128 requests for each of at most this many CTAs of a single-launch grid.
constexpr int kMaxBlockCtas = 256;
// Barrier words of the single launch's request tiles (at most kMaxBlockCtas
// tiles, 16 bytes each).
constexpr size_t kTileSyncBytes = 16 * kMaxBlockCtas;

// A per-range record of the running single launch (through L2 only).
__device__ __forceinline__ DraftPartial ld_part(const DraftPartial* p) {
  int4 v;
  asm volatile("ld.global.cg.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return DraftPartial{__int_as_float(v.x), __int_as_float(v.y), v.z, v.w};
}

// (R, S) += (R2, S2) for masses referenced to 2^R: aligned by an exact power
// of two (R = INT_MIN: nothing yet).
__device__ __forceinline__ void mass_add(int32_t& R, ff& S, int32_t R2, ff S2) {
  if (R2 == INT_MIN || !(S2.hi > 0.f)) return;
  if (R2 > R) {
    S = R == INT_MIN ? ff{0.f, 0.f} : ff_scale(S, pow2_nonpos(R - R2));
    R = R2;
  }
  S = ff_add(S, ff_scale(S2, pow2_nonpos(R2 - R)));
}

// One warp draws position k of request b in the single launch, from the
// masses of the CTAs' contiguous vocabulary ranges (parts: this request's
// per_m ranges, two group records each): the lanes own contiguous runs of
// ranges and scan them to the range holding u*Z (the lanes partition [0, Z)
// as in draw_request), that range's tiles are scanned to the crossing tile,
// and draw_in_tile finishes. Float pairs and exact powers of two throughout,
// as in draw_request; only the grouping of the sums differs.

constexpr int kRangesHeld = kMaxBlockCtas / 32;  // ranges per lane at most
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// One warp waits until the tags of all P ranges (tile_sync words of one
// request tile) have reached k + 1: each lane polls its own ranges' tags
// (relaxed loads, no warp-wide vote per try) and makes them acquires with a
// fence, then the warp meets. Returns false if the wait gave up.
__device__ __forceinline__ bool wait_range_tags(const uint32_t* tags, int P, int k, int lane) {
  const int per = (P + 31) / 32;
  const int p0 = min(lane * per, P), p1 = min(p0 + per, P);
  WaitClock clock;
  bool gave_up = false;
  for (;;) {
    bool mine = true;
#pragma unroll
    for (int i = 0; i < kRangesHeld; ++i)
      if (p0 + i < p1) mine = mine && ld_relaxed_gpu(tags + p0 + i) >= static_cast<uint32_t>(k + 1);
    if (mine) break;
    if (clock.expired()) {
      gave_up = true;
      break;
    }
    __nanosleep(32);
  }
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  __syncwarp();
  return !__any_sync(0xFFFFFFFFu, gave_up);
}

template <int kRec>  // records per range (one per epilogue group, or one combined)
__device__ __forceinline__ void draw_ranges(const DraftPickArgs& a, int b, int lane,
                                            const DraftPartial* parts, int per_m) {
  const int per = (per_m + 31) / 32;
  const int p0 = min(lane * per, per_m), p1 = min(p0 + per, per_m);
  const float u = a.uniforms[static_cast<size_t>(b) * a.gamma + a.k];
  int32_t rR[kRangesHeld];
  ff rS[kRangesHeld];
  int32_t Rl = INT_MIN;
  ff Sl{0.f, 0.f};
#pragma unroll
  for (int i = 0; i < kRangesHeld; ++i) {
    rR[i] = INT_MIN;
    rS[i] = ff{0.f, 0.f};
    if (p0 + i < p1) {
#pragma unroll
      for (int q = 0; q < kRec; ++q) {
        const DraftPartial d = ld_part(parts + kRec * (p0 + i) + q);
        mass_add(rR[i], rS[i], d.R, ff{d.hi, d.lo});
      }
      mass_add(Rl, Sl, rR[i], rS[i]);
    }
  }
  int32_t Rmax = Rl;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Rmax = max(Rmax, __shfl_xor_sync(0xFFFFFFFFu, Rmax, o));
  int y = 0;
  if (Rmax == INT_MIN || !(u >= 0.f && u < 1.f)) {
    if (lane == 0) set_status(a.status, DSPARK_ERR_BAD_DATA);
    publish_token(a, b, y, lane);
    return;
  }
  // level 1: the ranges
  const ff S = Rl == INT_MIN ? ff{0.f, 0.f} : ff_scale(Sl, pow2_nonpos(Rl - Rmax));
  const ff incl = warp_incl_scan_ff(S, lane);
  const ff Z = shfl_ff(incl, 31);
  const ff prev = shfl_up_ff(incl, 1);
  const ff excl = lane > 0 ? prev : ff{0.f, 0.f};
  const ff target = ff_mul(ff{u, 0.f}, Z);
  const uint32_t own = __ballot_sync(0xFFFFFFFFu, S.hi > 0.f && ff_cmp(excl, target) <= 0 &&
                                                        ff_cmp(target, incl) < 0);
  int ps = -1;
  ff before{0.f, 0.f};
  if (own && lane == __ffs(own) - 1) {  // walk this lane's ranges
    ff C = excl, Clast = excl;
    int plast = -1;
#pragma unroll
    for (int i = 0; i < kRangesHeld; ++i) {
      if (ps >= 0 || p0 + i >= p1 || rR[i] == INT_MIN || !(rS[i].hi > 0.f)) continue;
      const ff next = ff_add(C, ff_scale(rS[i], pow2_nonpos(rR[i] - Rmax)));
      if (ff_cmp(next, target) > 0) {
        ps = p0 + i;
        before = C;
      } else {
        plast = p0 + i;
        Clast = C;
        C = next;
      }
    }
    if (ps < 0) {  // rounding left the target past this lane's last range: take it
      ps = plast;
      before = Clast;
    }
  }
  const int ol = own ? __ffs(own) - 1 : 0;
  ps = own ? __shfl_sync(0xFFFFFFFFu, ps, ol) : -1;
  before = shfl_ff(before, ol);
  if (ps < 0) {  // no mass where the scan put the cut: the masses and the scan disagree
    if (lane == 0) set_status(a.status, DSPARK_ERR_BAD_DATA);
    publish_token(a, b, y, lane);
    return;
  }
  // level 2: the tiles of range ps, in order
  const DraftStat* st = a.stats + static_cast<size_t>(b) * a.n_tiles;
  const int t0 = range_begin(ps, a.n_tiles, per_m), t1 = range_begin(ps + 1, a.n_tiles, per_m);
  int g = -1, glast = -1;
  ff s_before{0.f, 0.f}, s_last{0.f, 0.f}, base = before;
  for (int c0 = t0; c0 < t1 && g < 0; c0 += 32) {
    const int t = c0 + lane;
    ff w{0.f, 0.f};
    if (t < t1) {
      const DraftStat d = ld_stat<true>(st + t);
      if (d.s > 0.f && d.R != INT_MIN) w = ff{d.s * pow2_nonpos(d.R - Rmax), 0.f};
    }
    const ff inc_t = ff_add(base, warp_incl_scan_ff(w, lane));
    const ff pre = shfl_up_ff(inc_t, 1);
    const ff exc_t = lane > 0 ? pre : base;
    const uint32_t cross = __ballot_sync(0xFFFFFFFFu, w.hi > 0.f && ff_cmp(inc_t, target) > 0);
    const uint32_t pos = __ballot_sync(0xFFFFFFFFu, w.hi > 0.f);
    if (cross) {
      const int l = __ffs(cross) - 1;
      g = c0 + l;
      s_before = shfl_ff(exc_t, l);
    } else if (pos) {
      const int l = 31 - __clz(pos);
      glast = c0 + l;
      s_last = shfl_ff(exc_t, l);
    }
    base = shfl_ff(inc_t, 31);
  }
  if (g < 0) {  // rounding: the range's last tile with mass
    g = glast;
    s_before = s_last;
  }
  if (g >= 0) y = draw_in_tile<true>(a, b, g, s_before, target, Rmax, lane);
  publish_token(a, b, y, lane);
}

__global__ void __launch_bounds__(kPickWarps * 32) k_draft_pick(const DraftPickArgs a) {
  const int b = blockIdx.x * kPickWarps + (threadIdx.x >> 5);
  if (b >= a.B) return;  // whole warps only
  draw_request<false>(a, b, threadIdx.x & 31);
}


// ---------------------------------------------------------------------------
// draft_tiles: the tile stage of positions [k_begin, k_end)
// ---------------------------------------------------------------------------
// Two instantiations. k_draft_step runs one position per launch and leaves the
// draw to k_draft_pick (G comes from the buffer the previous draw wrote).
// k_draft_block runs the whole block of gamma positions in one persistent
// kernel: the roles stay alive across the positions, so
// the producers stream W2 and U for position after position (the next
// position's tiles load while the current one draws), the tensor memory and
// the barriers stay set up, and the draws run inside the kernel after a
// barrier among the CTAs of each request tile (every statistic, range mass and
// row of the tile's requests at position k is written before any warp draws
// one of them; every G row of position k+1 is written before any CTA loads it:
// each drawing warp publishes its request's token with a flag, and a CTA waits
// only for its own rows; statistics and masses alternate between two buffers,
// so a CTA already writing position k+1's may not overwrite what a slower one
// still reads). Launched cooperatively (every CTA resident, one per
// SM), so no wait can be on a CTA that is not running; every spin is bounded.

// A diagnostic of the bounded waits: one thread runs a wait whose condition
// never comes true -- which 0: wait_or_flag on an mbarrier that no copy or
// thread completes (the waits of the pipelines' rings); which 1: grid_barrier
// for two CTAs in a grid of one (the drafter's barrier among the CTAs of a
// request tile) -- and the wait
// gives up, writes DSPARK_ERR_TIMEOUT to *status and the kernel returns.
__global__ void k_wait_selftest(int which, uint32_t* sync, int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  if (which == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    (void)wait_or_flag(&bar, 0, status);  // sets DSPARK_ERR_TIMEOUT when it gives up
  } else {
    uint32_t gen = ld_acquire_gpu(&sync[1]);
    if (!grid_barrier(sync, 2u, gen)) set_status(status, DSPARK_ERR_TIMEOUT);
  }
}


struct DraftBlockArgs {
  DraftStepArgs s;     // s.k unused; s.stats: the statistics (of even positions)
  DraftPickArgs p;     // p.k and p.stats set per position
  int32_t k_begin, k_end;       // the positions this launch runs
  const uint16_t* G;            // per-launch path: G = W1[x_{k-1}] written by the previous draw
  DraftStat* stats1;            // single launch: the statistics of odd positions
  const int32_t* anchors;       // x_0
  uint32_t* sync;               // [2]
  unsigned long long* ready;    // [B]
  uint32_t* tile_sync;          // [n_m][4]: a barrier (count, generation) per request tile
  DraftPartial* parts;          // [2][n_m * 128][per_m]: per-range masses by position parity
};

template <bool kBlock>
__device__ __forceinline__ void draft_tiles(const CUtensorMap& mapW, const CUtensorMap& mapU,
                                            const CUtensorMap& mapL, const DraftBlockArgs& ba) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  DraftBars* bars = reinterpret_cast<DraftBars*>(smem + kOffBar);
  const DraftStepArgs& a = ba.s;
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The CTAs that share a vocabulary range (one per request tile) read the
  // same W2 tiles. In the single launch every CTA holds an SM of its own
  // (one fits per SM), so when the grid covers every SM id the SM id itself
  // is a permutation of the CTA indices: neighbouring ids (the two SMs of a
  // TPC) then take the same range. Block indices are dealt across the GPU, so
  // without this the pair of a range sits on two distant SMs (measured about
  // 1% slower per block).
  uint32_t cta = blockIdx.x;
  if (kBlock) {
    uint32_t smid, nsmid;
    asm("mov.u32 %0, %%smid;" : "=r"(smid));
    asm("mov.u32 %0, %%nsmid;" : "=r"(nsmid));
    if (nsmid == gridDim.x && smid < nsmid) cta = smid;
  }
  const int m_tile = static_cast<int>(cta) % a.n_m;
  const int p = static_cast<int>(cta) / a.n_m;  // this CTA's vocabulary range in its request tile
  const int lo = range_begin(p, a.n_tiles, a.per_m), hi = range_begin(p + 1, a.n_tiles, a.per_m);
  const int n_local = hi - lo;
  const int KC = a.r / kDK;
  const int k0 = ba.k_begin;
  const int npos = ba.k_end - ba.k_begin;  // positions of this launch
  // position k's t-th vocabulary tile of this CTA: its contiguous range, odd
  // positions backwards (a position starts on the W2 tiles the previous one
  // read last; the CTAs of the other request tiles walk the same ranges)
  auto tile_of = [&](int k, int t) { return (k & 1) ? hi - 1 - t : lo + t; };

  if (threadIdx.x == 0) {
    mbar_init(&bars->a_full, kDEpiWarps);
    for (int s = 0; s < kDStages; ++s) {
      mbar_init(&bars->w_full[s], 1);
      mbar_init(&bars->w_empty[s], 1);
    }
    for (int s = 0; s < kDSlots; ++s) {
      mbar_init(&bars->u_full[s], 1);
      mbar_init(&bars->u_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_empty[i], 4);
      mbar_init(&bars->st_ready[i], 4);
    }
    mbar_init(&bars->mma_done, 1);
    mbar_init(&bars->epi_done, kDEpiWarps);
    mbar_init(&bars->step_go, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ---------------- W2 producer: every position's chunks, in order ----------------
    if (lane == 0) {
      tma_prefetch_map(&mapW);
      const uint64_t pol_keep = policy_evict_last();
      const int total = npos * n_local * KC;
      bool ok = true;
      int nq = 0;
      for (int q = 0; q < total; ++q) {
        const int tg = q / KC, c = q % KC, s = q % kDStages;
        if (q >= kDStages) {
          ok = wait_or_flag(&bars->w_empty[s], ((q / kDStages) - 1) & 1, a.status);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(&bars->w_full[s], kBoxW);
        tma_load_2d(smem + kOffW + s * kBoxW, &mapW, c * kDK,
                    tile_of(k0 + tg / n_local, tg % n_local) * kDN, &bars->w_full[s], pol_keep);
        nq = q + 1;
      }
      if (!ok)
        for (int q = nq - kDStages > 0 ? nq - kDStages : 0; q < nq; ++q)
          mbar_wait(&bars->w_full[q % kDStages], (q / kDStages) & 1);
    }
  } else if (warp == kDWarpU) {
    // ---------------- U producer: every position's tiles, in order ----------------
    if (lane == 0) {
      tma_prefetch_map(&mapU);
      const uint64_t pol_stream = policy_evict_first();
      const int total = npos * n_local;
      bool ok = true;
      int nu = 0;
      for (int tg = 0; tg < total; ++tg) {
        const int slot = tg % kDSlots;
        if (tg >= kDSlots) {
          ok = wait_or_flag(&bars->u_empty[slot], ((tg / kDSlots) - 1) & 1, a.status);
          if (!ok) break;
        }
        const int k = k0 + tg / n_local;
        const int v0 = tile_of(k, tg % n_local) * kDN;
        uint8_t* dst = smem + kOffU + slot * 2 * kBoxU;
        mbar_arrive_expect_tx(&bars->u_full[slot], 2 * kBoxU);
        tma_load_3d(dst, &mapU, v0, k, m_tile * kDM, &bars->u_full[slot], pol_stream);
        tma_load_3d(dst + kBoxU, &mapU, v0 + kDK, k, m_tile * kDM, &bars->u_full[slot],
                    pol_stream);
        nu = tg + 1;
      }
      if (!ok)
        for (int t = nu - kDSlots > 0 ? nu - kDSlots : 0; t < nu; ++t)
          mbar_wait(&bars->u_full[t % kDSlots], (t / kDSlots) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      for (int j = 0; j < npos && ok && n_local > 0; ++j) {
        ok = wait_or_flag(&bars->a_full, j & 1, a.status);  // G of position k0 + j in tensor memory
        if (!ok) break;
        tc_fence_after();
        for (int t = 0; t < n_local && ok; ++t) {
          const int tg = j * n_local + t;
          const int acc = tg & 1;
          if (tg >= 2) {
            ok = wait_or_flag(&bars->acc_empty[acc], ((tg >> 1) - 1) & 1, a.status);
            if (!ok) break;
            tc_fence_after();
          }
          const uint32_t d = tmem + acc * kDN;
          for (int c = 0; c < KC && ok; ++c) {
            const int q = tg * KC + c, s = q % kDStages;
            ok = wait_or_flag(&bars->w_full[s], (q / kDStages) & 1, a.status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t w_base = sbase + kOffW + s * kBoxW;
#pragma unroll
            for (int kk = 0; kk < kDK / 16; ++kk)
              tc_mma_ts(d, tmem + kColG + c * (kDK / 2) + kk * 8, sdesc_sw128(w_base + 32 * kk),
                        kIdesc, (c | kk) != 0);
            tc_commit(&bars->w_empty[s]);
          }
          if (ok) tc_commit(&bars->acc_full[acc]);
        }
      }
      tc_commit(&bars->mma_done);
      wait_or_flag(&bars->mma_done, 0, a.status);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue + draw warps ----------------
    const int ew = warp - 2;          // 0..7
    const int grp = ew >> 2;
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const int b = m_tile * kDM + m;
    const bool row_ok = b < a.B;
    const bool leader = (warp == 2 + 4 * grp) && lane == 0;
    const bool syncer = warp == 2 && lane == 0;  // takes part in the tile barriers
    const uint64_t pol_out = policy_evict_first();
    uint32_t gen = 0;
    // the CTAs of one request tile synchronise among themselves: a position's
    // draws read only that tile's statistics and range masses, and its next
    // position waits only on that tile's tokens
    // (the per-launch kernel has no barrier words and never touches them)
    uint32_t* const tbar = kBlock ? ba.tile_sync + 4 * m_tile : nullptr;
    if constexpr (kBlock)
      if (syncer) gen = ld_acquire_gpu(&tbar[1]);
    int jg = 0;        // tiles this group has finished (all positions)
    int uses = 0;      // epi_done / step_go phases used so far
    bool ok = true;
    // the request tile's barrier: the CTA's eight warps report, one thread
    // crosses with the tile's other CTAs, all go on
    auto tile_barrier = [&]() {
      if (lane == 0) mbar_arrive(&bars->epi_done);
      bool good = true;
      if (syncer) {
        good = wait_or_flag(&bars->epi_done, uses & 1, a.status) &&
               grid_barrier(tbar, static_cast<uint32_t>(a.per_m), gen);
        if (!good) set_status(a.status, DSPARK_ERR_TIMEOUT);
        mbar_arrive(&bars->step_go);
      }
      good = wait_or_flag(&bars->step_go, uses & 1, a.status) && good;
      ++uses;
      return __all_sync(0xFFFFFFFFu, good);
    };
    for (int j = 0; j < npos && ok; ++j) {
      const int k = k0 + j;
      // G = W1[x_{k-1}] of this request tile into tensor memory: group g
      // writes K elements [128 g, 128 g + 128) of row m (rows past the batch:
      // 0). Single launch: x_0 is the anchor and x_{k-1} comes with the flag its
      // drawing warp published; per launch: the row the previous kernel wrote
      int x = 0;
      if constexpr (kBlock) {
        bool r_ok = true;
        if (row_ok) {
          if (k == 0) {
            x = ba.anchors[b];
            if (x < 0 || x >= a.V) {
              set_status(a.status, DSPARK_ERR_BAD_DATA);
              x = 0;
            }
          } else {
            WaitClock clock;
            unsigned long long f;
            while (((f = ld_acquire_gpu64(&ba.ready[b * kReadyStride])) >> 32) < static_cast<unsigned>(k)) {
              if (clock.expired()) {
                r_ok = false;
                break;
              }
              __nanosleep(32);
            }
            x = static_cast<int>(static_cast<uint32_t>(f));
          }
        }
        if (!__all_sync(0xFFFFFFFFu, r_ok)) {
          set_status(a.status, DSPARK_ERR_TIMEOUT);
          break;
        }
      }
      {
        const uint16_t* row = kBlock ? ba.p.W1 + static_cast<size_t>(x) * a.r
                                     : ba.G + static_cast<size_t>(b) * a.r;
        const uint4* src = reinterpret_cast<const uint4*>(row);
        const int c0 = grp * 2;
        const int nc = KC - c0 < 0 ? 0 : (KC - c0 > 2 ? 2 : KC - c0);
        uint32_t w[2][32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 v = row_ok && cc < nc ? __ldg(src + (c0 + cc) * 8 + i)
                                              : make_uint4(0u, 0u, 0u, 0u);
            w[cc][4 * i] = v.x;
            w[cc][4 * i + 1] = v.y;
            w[cc][4 * i + 2] = v.z;
            w[cc][4 * i + 3] = v.w;
          }
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
          if (cc < nc)
            tmem_st32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kColG + (c0 + cc) * 32,
                      w[cc]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->a_full);
      }
      // this position's tiles: tile tg of the block goes to group tg & 1; the
      // single launch also sums each request's mass over the group's tiles
      int32_t Rp = INT_MIN;
      ff Sp{0.f, 0.f};
      for (int t = 0; t < n_local; ++t) {
        const int tg = j * n_local + t;
        if ((tg & 1) != grp) continue;
        const int n = tile_of(k, t);
        const int v0 = n * kDN;
        const int slot = tg % kDSlots;
        const uint32_t ubase = sbase + kOffU + slot * 2 * kBoxU;
        bool w_ok = wait_or_flag(&bars->acc_full[grp], (tg >> 1) & 1, a.status);
        w_ok = w_ok && wait_or_flag(&bars->u_full[slot], (tg / kDSlots) & 1, a.status);
        if (!__all_sync(0xFFFFFFFFu, w_ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + grp * kDN;
        int32_t R;
        float total;
        bool inf_seen = false;
        if (v0 + kDN <= a.V)
          epi_tile<true>(taddr, ubase, m, v0, a.V, a.ep, R, total, inf_seen,
                         &bars->acc_empty[grp], lane);
        else
          epi_tile<false>(taddr, ubase, m, v0, a.V, a.ep, R, total, inf_seen,
                          &bars->acc_empty[grp], lane);
        const bool bad = inf_seen || total != total;
        if (row_ok) {
          if (bad) set_status(a.status, DSPARK_ERR_BAD_DATA);
          ((kBlock && (k & 1)) ? ba.stats1 : a.stats)[static_cast<size_t>(b) * a.n_tiles + n] =
              DraftStat{bad ? 0.f : total, bad ? INT_MIN : R};
        }
        if constexpr (kBlock)
          if (!bad && total > 0.f) mass_add(Rp, Sp, R, ff{total, 0.f});
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->st_ready[grp]);
        if (leader && wait_or_flag(&bars->st_ready[grp], jg & 1, a.status)) {
          tma_store_3d(&mapL, smem + kOffU + slot * 2 * kBoxU, v0, k, m_tile * kDM, pol_out);
          if (v0 + kDK < a.V)
            tma_store_3d(&mapL, smem + kOffU + slot * 2 * kBoxU + kBoxU, v0 + kDK, k,
                         m_tile * kDM, pol_out);
          bulk_commit();
          bulk_wait_read<0>();
          mbar_arrive(&bars->u_empty[slot]);
        }
        ++jg;
        __syncwarp();
      }
      if (!ok) break;
      if constexpr (!kBlock) break;  // one position; the draw is the next kernel
      if (row_ok)  // this group's share of the request's mass over the CTA's range
        ba.parts[((static_cast<size_t>(k & 1) * a.n_m * kDM + b) * a.per_m + p) * 2 + grp] =
            DraftPartial{Sp.hi, Sp.lo, Rp, 0};
      // the rows of this position are in memory (stores complete, visible to
      // the generic proxy of every CTA) and so are the statistics
      if (leader) {
        bulk_wait<0>();
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      __threadfence();
      if (!tile_barrier()) {
        ok = false;
        break;
      }
      // the draws: one warp per request, spread over the request tile's CTAs
      DraftPickArgs pa = ba.p;
      pa.k = k;
      pa.stats = (k & 1) ? ba.stats1 : a.stats;
      pa.ready = ba.ready;
      // one request per epilogue warp, from the ranges' masses
      const DraftPartial* parts_k =
          ba.parts + static_cast<size_t>(k & 1) * a.n_m * kDM * a.per_m * 2;
      for (int i = ew * a.per_m + p; i < kDM; i += kDEpiWarps * a.per_m) {
        const int rq = m_tile * kDM + i;
        if (rq >= a.B) break;
        draw_ranges<2>(pa, rq, lane, parts_k + static_cast<size_t>(rq) * a.per_m * 2, a.per_m);
      }
    }
    if (leader) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One position per launch (the per-launch path: grids that cannot be resident
// at once, and the timed entry point); the draw is k_draft_pick.
__global__ void __launch_bounds__(kDThreads, 1)
    k_draft_step(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapU,
                 const __grid_constant__ CUtensorMap mapL, const DraftBlockArgs ba) {
  draft_tiles<false>(mapW, mapU, mapL, ba);
}

// The whole block in one cooperative launch, draws included.
__global__ void __launch_bounds__(kDThreads, 1)
    k_draft_block(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapU,
                  const __grid_constant__ CUtensorMap mapL, const DraftBlockArgs ba) {
  draft_tiles<true>(mapW, mapU, mapL, ba);
}

// ---------------------------------------------------------------------------
// k_draft_pair: the whole block for two request tiles (128 < B <= 256) in one
// cooperative launch: most CTAs stream both request tiles, a few only draw
// ---------------------------------------------------------------------------
// In k_draft_block the CTAs of a request tile stream that tile's vocabulary
// ranges, then wait at the tile's barrier, draw and load the next G while the
// memory system idles. Here each streaming CTA owns one contiguous vocabulary
// range for both request tiles and alternates: position k's tiles of request
// tile 0, then those of request tile 1 (walking the range backwards, so that
// it starts on the W2 tiles just read), then position k + 1's of tile 0, ...
// A request tile's end of a position runs beside the other tile's streaming:
// the epilogue leaves its range masses (one record per request and CTA) behind
// and streams on; a release warp publishes the CTA's tag for (tile, position)
// once the rows, statistics and records are in memory. The draws run on CTAs
// of their own (kPDrawCtas of them, one warp per request of a tile), which
// read the tags of every range and then draw; on the streaming SMs the draws'
// chains of dependent loads would compete with the streams. The streaming
// CTAs' four G warps wait for the tile's tokens and write its next
// G = W1[x_k] into tensor memory. No CTA waits at a grid-wide barrier. Tensor
// memory: two f32 accumulators of 128 columns, then G of request tile 0 and of
// request tile 1 (r / 2 columns each): 512 columns at r = 256.
// W2 ring and U / L tile slots: 5 stages of W2 chunks (1.25 vocabulary tiles)
// and 4 tile slots measured 1.3% faster on 256 x 16 x 129,280 than 7 and 3
// (two slots are held by the epilogue groups, so 4 keeps two loading), and 3
// and 5 slower
constexpr int kPStages = 5;
constexpr int kPSlots = 4;
constexpr int kPGWarps = 4;     // G loaders: one per lane quarter of tensor memory
constexpr int kPWarpU = 2 + kDEpiWarps;      // the U producer's warp
constexpr int kPWarpG = kPWarpU + 1;         // the G warps' first
constexpr int kPWarpRel = kPWarpG + kPGWarps;  // the release warp
// draw CTAs beside the streaming ones: with 16 warps each, 8 give one warp per
// request of a tile (measured on 256 x 16 x 129,280: 0.69 ms per block with 8,
// 0.76 with 4 or 6, 0.72-0.73 with 10 or 16)
constexpr int kPDrawCtas = 8;
constexpr int kPThreads = (kPWarpRel + 1) * 32;
constexpr uint32_t kPOffU = kPStages * kBoxW;
constexpr uint32_t kPOffPart = kPOffU + kPSlots * 2 * kBoxU;  // [request tile][group][row]
constexpr uint32_t kPOffBar = kPOffPart + 2 * 2 * kDM * sizeof(DraftPartial);
constexpr uint32_t kPairSmem = kPOffBar + 512 + 1024;
static_assert(kPairSmem <= 232448, "shared memory of k_draft_pair");
static_assert(kColG + 2 * (DSPARK_DRAFT_MAX_RANK / 2) <= kTmemCols, "tensor memory of k_draft_pair");
static_assert(2 * kMaxBlockCtas * 4 <= kTileSyncBytes, "tags of k_draft_pair");

struct PairBars {
  uint64_t a_full[2];  // G of request tile g in tensor memory (one arrival per G warp)
  uint64_t w_full[kPStages], w_empty[kPStages];
  uint64_t u_full[kPSlots], u_empty[kPSlots];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t st_ready[2];  // a group's rows are in shared memory, ready to store
  uint64_t mma_done;
  uint64_t epi_done[2];  // the epilogue finished request tile g's tiles of a position
  uint32_t tmem_base;
};
static_assert(sizeof(PairBars) <= 512, "barrier block of k_draft_pair");

// The eight epilogue warps of the CTA (256 threads) meet: named barrier 1.
__device__ __forceinline__ void epi_warps_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDEpiWarps * 32) : "memory");
}

// G of request tile g into tensor memory, rows of this warp's lane quarter
// (request g * 128 + 32 * quarter + lane): W1[x] for the token x the row's
// request drew at position k - 1 (the anchor at k = 0), zero past the batch.
// Returns false if a wait gave up.
__device__ __forceinline__ bool pair_load_g(const DraftBlockArgs& ba, int g, int k, uint32_t tmem,
                                            int quarter, int lane) {
  const DraftStepArgs& a = ba.s;
  const int b = g * kDM + quarter * 32 + lane;
  const bool row_ok = b < a.B;
  int x = 0;
  bool r_ok = true;
  if (row_ok) {
    if (k == 0) {
      x = ba.anchors[b];
      if (x < 0 || x >= a.V) {
        set_status(a.status, DSPARK_ERR_BAD_DATA);
        x = 0;
      }
    } else {
      // the flag carries the token; W1 is an input, so a relaxed read suffices
      WaitClock clock;
      unsigned long long f;
      for (;;) {
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(f) : "l"(&ba.ready[b * kReadyStride]) : "memory");
        if ((f >> 32) >= static_cast<unsigned>(k)) break;
        if (clock.expired()) {
          r_ok = false;
          break;
        }
        __nanosleep(32);
      }
      x = static_cast<int>(static_cast<uint32_t>(f));
    }
  }
  if (!__all_sync(0xFFFFFFFFu, r_ok)) {
    set_status(a.status, DSPARK_ERR_TIMEOUT);
    return false;
  }
  const uint4* src = reinterpret_cast<const uint4*>(ba.p.W1 + static_cast<size_t>(x) * a.r);
  const int KC = a.r / kDK;
  const uint32_t t0 = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kColG +
                      static_cast<uint32_t>(g) * (DSPARK_DRAFT_MAX_RANK / 2);
  // two 64-element chunks (32 columns each) per round: both chunks' loads are
  // in flight before the first store to tensor memory (a store is ordered
  // after every earlier load of the warp)
  for (int c = 0; c < KC; c += 2) {
    const bool two = c + 1 < KC;
    uint32_t w0[32], w1[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 v = row_ok ? __ldg(src + c * 8 + i) : make_uint4(0u, 0u, 0u, 0u);
      w0[4 * i] = v.x;
      w0[4 * i + 1] = v.y;
      w0[4 * i + 2] = v.z;
      w0[4 * i + 3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 v = row_ok && two ? __ldg(src + (c + 1) * 8 + i) : make_uint4(0u, 0u, 0u, 0u);
      w1[4 * i] = v.x;
      w1[4 * i + 1] = v.y;
      w1[4 * i + 2] = v.z;
      w1[4 * i + 3] = v.w;
    }
    __syncwarp();
    tmem_st32(t0 + c * 32, w0);
    if (two) tmem_st32(t0 + (c + 1) * 32, w1);
  }
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  return true;
}

__global__ void __launch_bounds__(kPThreads, 1)
    k_draft_pair(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapU,
                 const __grid_constant__ CUtensorMap mapL, const DraftBlockArgs ba) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  PairBars* bars = reinterpret_cast<PairBars*>(smem + kPOffBar);
  DraftPartial* part = reinterpret_cast<DraftPartial*>(smem + kPOffPart);
  const DraftStepArgs& a = ba.s;
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = a.per_m;  // streaming CTAs: vocabulary ranges; the rest draw
  const int p = blockIdx.x;
  if (p >= P) {
    // ---------------- draw CTA: one warp per request of each (tile, position) ----------------
    // (no tensor memory, barriers or shared memory: it reads the tags, the
    // range records and statistics, and the rows of the tile it picks)
    const int n_draw_warps = (static_cast<int>(gridDim.x) - P) * (kPThreads / 32);
    const int wid = (p - P) * (kPThreads / 32) + warp;
    const size_t n_req = static_cast<size_t>(a.n_m) * kDM;
    // warp 0 waits for the tags of (tile, position) and takes the acquire;
    // the CTA's barrier then orders every warp's loads after it (one poller
    // per CTA: every warp starts together, and 16 times fewer polls)
    __shared__ int sh_gave_up[2];  // by parity: rewritten two barriers later
    for (int it = 0; it < 2 * a.gamma; ++it) {
      const int k = it >> 1, g = it & 1;
      if (warp == 0) {
        const bool got = wait_range_tags(ba.tile_sync + g * kMaxBlockCtas, P, k, lane);
        if (lane == 0) sh_gave_up[it & 1] = got ? 0 : 1;
      }
      __syncthreads();
      if (sh_gave_up[it & 1]) {
        if (threadIdx.x == 0) set_status(a.status, DSPARK_ERR_TIMEOUT);
        break;
      }
      DraftPickArgs pa = ba.p;
      pa.k = k;
      pa.stats = (k & 1) ? ba.stats1 : a.stats;
      pa.ready = ba.ready;
      pa.relaxed_flag = true;
      for (int i = wid; i < kDM; i += n_draw_warps) {
        const int rq = g * kDM + i;
        if (rq >= a.B) break;
        draw_ranges<1>(pa, rq, lane, ba.parts + (static_cast<size_t>(k & 1) * n_req + rq) * P, P);
      }
    }
    return;
  }
  const int lo = range_begin(p, a.n_tiles, P), hi = range_begin(p + 1, a.n_tiles, P);
  const int n_local = hi - lo;
  const int KC = a.r / kDK;
  const int gamma = a.gamma;
  const size_t n_req = static_cast<size_t>(a.n_m) * kDM;
  uint32_t* const tags = ba.tile_sync;  // [2][kMaxBlockCtas]: (tile, CTA) -> position + 1
  // request tile g's t-th vocabulary tile of this range: tile 0 forwards, tile
  // 1 backwards (so each starts on the W2 tiles the other read last)
  auto tile_of = [&](int g, int t) { return g ? hi - 1 - t : lo + t; };
  // tile index tg over (position, request tile, t): its position and request tile
  auto pos_of = [&](int tg) { return tg / (2 * n_local); };
  auto rt_of = [&](int tg) { return (tg / n_local) & 1; };

  if (threadIdx.x == 0) {
    for (int g = 0; g < 2; ++g) {
      mbar_init(&bars->a_full[g], kPGWarps);
      mbar_init(&bars->epi_done[g], kDEpiWarps);
    }
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&bars->w_full[s], 1);
      mbar_init(&bars->w_empty[s], 1);
    }
    for (int s = 0; s < kPSlots; ++s) {
      mbar_init(&bars->u_full[s], 1);
      mbar_init(&bars->u_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_empty[i], 4);
      mbar_init(&bars->st_ready[i], 4);
    }
    mbar_init(&bars->mma_done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const int total_tiles = gamma * 2 * n_local;

  if (warp == 0) {
    // ---------------- W2 producer: the chunks of every tile, in order ----------------
    if (lane == 0) {
      tma_prefetch_map(&mapW);
      const uint64_t pol_keep = policy_evict_last();
      const int total = total_tiles * KC;
      bool ok = true;
      int nq = 0;
      for (int q = 0; q < total; ++q) {
        const int tg = q / KC, c = q % KC, s = q % kPStages;
        if (q >= kPStages) {
          ok = wait_or_flag(&bars->w_empty[s], ((q / kPStages) - 1) & 1, a.status);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(&bars->w_full[s], kBoxW);
        tma_load_2d(smem + s * kBoxW, &mapW, c * kDK, tile_of(rt_of(tg), tg % n_local) * kDN,
                    &bars->w_full[s], pol_keep);
        nq = q + 1;
      }
      if (!ok)
        for (int q = nq - kPStages > 0 ? nq - kPStages : 0; q < nq; ++q)
          mbar_wait(&bars->w_full[q % kPStages], (q / kPStages) & 1);
    }
  } else if (warp == kPWarpU) {
    // ---------------- U producer: every tile, in order ----------------
    if (lane == 0) {
      tma_prefetch_map(&mapU);
      const uint64_t pol_stream = policy_evict_first();
      bool ok = true;
      int nu = 0;
      for (int tg = 0; tg < total_tiles; ++tg) {
        const int slot = tg % kPSlots;
        if (tg >= kPSlots) {
          ok = wait_or_flag(&bars->u_empty[slot], ((tg / kPSlots) - 1) & 1, a.status);
          if (!ok) break;
        }
        const int g = rt_of(tg);
        const int v0 = tile_of(g, tg % n_local) * kDN;
        uint8_t* dst = smem + kPOffU + slot * 2 * kBoxU;
        mbar_arrive_expect_tx(&bars->u_full[slot], 2 * kBoxU);
        tma_load_3d(dst, &mapU, v0, pos_of(tg), g * kDM, &bars->u_full[slot], pol_stream);
        tma_load_3d(dst + kBoxU, &mapU, v0 + kDK, pos_of(tg), g * kDM, &bars->u_full[slot],
                    pol_stream);
        nu = tg + 1;
      }
      if (!ok)
        for (int t = nu - kPSlots > 0 ? nu - kPSlots : 0; t < nu; ++t)
          mbar_wait(&bars->u_full[t % kPSlots], (t / kPSlots) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      for (int j = 0; j < gamma && ok; ++j)
        for (int g = 0; g < 2 && ok; ++g) {
          ok = wait_or_flag(&bars->a_full[g], j & 1, a.status);  // G of (g, j) in tensor memory
          if (!ok) break;
          tc_fence_after();
          const uint32_t a_col = tmem + kColG + static_cast<uint32_t>(g) * (DSPARK_DRAFT_MAX_RANK / 2);
          for (int t = 0; t < n_local && ok; ++t) {
            const int tg = (j * 2 + g) * n_local + t;
            const int acc = tg & 1;
            if (tg >= 2) {
              ok = wait_or_flag(&bars->acc_empty[acc], ((tg >> 1) - 1) & 1, a.status);
              if (!ok) break;
              tc_fence_after();
            }
            const uint32_t d = tmem + acc * kDN;
            for (int c = 0; c < KC && ok; ++c) {
              const int q = tg * KC + c, s = q % kPStages;
              ok = wait_or_flag(&bars->w_full[s], (q / kPStages) & 1, a.status);
              if (!ok) break;
              tc_fence_after();
              const uint32_t w_base = sbase + s * kBoxW;
#pragma unroll
              for (int kk = 0; kk < kDK / 16; ++kk)
                tc_mma_ts(d, a_col + c * (kDK / 2) + kk * 8, sdesc_sw128(w_base + 32 * kk), kIdesc,
                          (c | kk) != 0);
              tc_commit(&bars->w_empty[s]);
            }
            if (ok) tc_commit(&bars->acc_full[acc]);
          }
        }
      tc_commit(&bars->mma_done);
      wait_or_flag(&bars->mma_done, 0, a.status);
    }
    __syncwarp();
  } else if (warp < kPWarpU) {
    // ---------------- epilogue: every tile, in order ----------------
    const int ew = warp - 2;  // 0..7
    const int grp = ew >> 2;
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const bool leader = (warp == 2 + 4 * grp) && lane == 0;
    const uint64_t pol_out = policy_evict_first();
    int jg = 0;  // tiles this group has finished
    bool ok = true;
    for (int j = 0; j < gamma && ok; ++j) {
      const int k = j;
      DraftStat* st_k = (k & 1) ? ba.stats1 : a.stats;
      for (int g = 0; g < 2 && ok; ++g) {
        const int b = g * kDM + m;
        const bool row_ok = b < a.B;
        int32_t Rp = INT_MIN;
        ff Sp{0.f, 0.f};
        for (int t = 0; t < n_local; ++t) {
          const int tg = (j * 2 + g) * n_local + t;
          if ((tg & 1) != grp) continue;
          const int n = tile_of(g, t);
          const int v0 = n * kDN;
          const int slot = tg % kPSlots;
          const uint32_t ubase = sbase + kPOffU + slot * 2 * kBoxU;
          bool w_ok = wait_or_flag(&bars->acc_full[grp], (tg >> 1) & 1, a.status);
          w_ok = w_ok && wait_or_flag(&bars->u_full[slot], (tg / kPSlots) & 1, a.status);
          if (!__all_sync(0xFFFFFFFFu, w_ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + grp * kDN;
          int32_t R;
          float total;
          bool inf_seen = false;
          if (v0 + kDN <= a.V)
            epi_tile<true>(taddr, ubase, m, v0, a.V, a.ep, R, total, inf_seen,
                           &bars->acc_empty[grp], lane);
          else
            epi_tile<false>(taddr, ubase, m, v0, a.V, a.ep, R, total, inf_seen,
                            &bars->acc_empty[grp], lane);
          const bool bad = inf_seen || total != total;
          if (row_ok) {
            if (bad) set_status(a.status, DSPARK_ERR_BAD_DATA);
            st_k[static_cast<size_t>(b) * a.n_tiles + n] =
                DraftStat{bad ? 0.f : total, bad ? INT_MIN : R};
            if (!bad && total > 0.f) mass_add(Rp, Sp, R, ff{total, 0.f});
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->st_ready[grp]);
          if (leader && wait_or_flag(&bars->st_ready[grp], jg & 1, a.status)) {
            tma_store_3d(&mapL, smem + kPOffU + slot * 2 * kBoxU, v0, k, g * kDM, pol_out);
            if (v0 + kDK < a.V)
              tma_store_3d(&mapL, smem + kPOffU + slot * 2 * kBoxU + kBoxU, v0 + kDK, k, g * kDM,
                           pol_out);
            bulk_commit();
            bulk_wait_read<0>();
            mbar_arrive(&bars->u_empty[slot]);
          }
          ++jg;
          __syncwarp();
        }
        if (!ok) break;
        // the row's mass over the range: group 1 hands its share over through
        // shared memory, group 0 writes the record; the rows of (g, k) are
        // stored before the release warp publishes the CTA's tag
        if (grp == 1) part[g * kDM + m] = DraftPartial{Sp.hi, Sp.lo, Rp, 0};
        if (leader) {
          bulk_wait<0>();
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        epi_warps_sync();
        if (grp == 0 && row_ok) {
          const DraftPartial o = part[g * kDM + m];
          mass_add(Rp, Sp, o.R, ff{o.hi, o.lo});
          ba.parts[(static_cast<size_t>(k & 1) * n_req + b) * P + p] =
              DraftPartial{Sp.hi, Sp.lo, Rp, 0};
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->epi_done[g]);
      }
    }
    if (leader) bulk_wait<0>();
  } else if (warp == kPWarpRel) {
    // ---------------- release warp: publishes the CTA's tag of (g, k) ----------------
    if (lane == 0) {
      bool ok = true;
      for (int j = 0; j < gamma && ok; ++j)
        for (int g = 0; g < 2 && ok; ++g) {
          ok = wait_or_flag(&bars->epi_done[g], j & 1, a.status);
          if (!ok) break;
          // a release at GPU scope: the epilogue's rows, statistics and records,
          // which this thread saw through epi_done, are visible before the tag
          st_release_gpu(&tags[g * kMaxBlockCtas + p], static_cast<uint32_t>(j + 1));
        }
    }
    __syncwarp();
  } else {
    // ---------------- G warps: each request tile's next G ----------------
    const int quarter = warp & 3;
    bool ok = true;
    for (int g = 0; g < 2 && ok; ++g) {  // G of position 0: W1 at the anchors
      ok = pair_load_g(ba, g, 0, tmem, quarter, lane);
      if (ok && lane == 0) mbar_arrive(&bars->a_full[g]);
    }
    for (int j = 0; j + 1 < gamma && ok; ++j)
      for (int g = 0; g < 2 && ok; ++g) {
        // G of (g, j + 1), once this CTA's MMAs of (g, j) have completed (its
        // epilogue finished with their accumulators) and the tile's tokens x_j
        // are drawn (pair_load_g waits for them)
        ok = __all_sync(0xFFFFFFFFu, wait_or_flag(&bars->epi_done[g], j & 1, a.status));
        ok = ok && pair_load_g(ba, g, j + 1, tmem, quarter, lane);
        if (ok && lane == 0) mbar_arrive(&bars->a_full[g]);
      }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct DraftDevice {
  bool ready = false;
  bool coop = false;
  int sms = 0;
};
std::mutex g_draft_mutex;

// The drafter's kernels are launched without programmatic dependent launch:
// measured on this pair, that attribute made a 16-position block about 70%
// slower (1.70 ms against 1.01 ms at 256 x 16 x 129,280), wherever the
// kernels triggered their dependents.
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
DraftDevice g_draft_dev[128];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int draft_setup(int& sms, bool& coop) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return DSPARK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_draft_mutex);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return DSPARK_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  DraftDevice& d = g_draft_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    if (cudaFuncSetAttribute(k_draft_step, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kDraftSmem)) != cudaSuccess ||
        cudaFuncSetAttribute(k_draft_block, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kDraftSmem)) != cudaSuccess ||
        cudaFuncSetAttribute(k_draft_pair, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kPairSmem)) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    int coop = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    d.coop = coop != 0;
    d.ready = true;
  }
  sms = d.sms;
  coop = d.coop;
  return DSPARK_OK;
}

// A bf16 tensor map in the 128-byte swizzled layout: dims[0] innermost.
bool encode_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                  const_cast<void*>(base), dims, strides_bytes, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ExpParams draft_exp_params(float temperature) {
  ExpParams ep;
  ep.c_d = 1.4426950408889634 / static_cast<double>(temperature);  // log2(e) / T
  float hi = static_cast<float>(ep.c_d);
  if (static_cast<double>(hi) > ep.c_d) hi = std::nextafter(hi, 0.0f);
  ep.c_hi = hi;
  ep.c_lo = static_cast<float>(ep.c_d - static_cast<double>(hi));
  if (!(ep.c_lo > 0.0f)) ep.c_lo = 1e-30f;  // keeps c_lo * (-inf) = -inf
  return ep;
}

int draft_entry(const void* base_logits, const void* w1, const void* w2t, const int32_t* anchors,
                const float* uniforms, float temperature, int32_t B, int32_t gamma, int64_t V,
                int32_t r, void* draft_logits, int32_t* draft_tokens, int32_t* device_status,
                void* workspace, size_t workspace_bytes, cudaStream_t stream, cudaEvent_t* ev) {
  if (B < 0 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || V < 8 || V % 8 != 0 ||
      V > (int64_t)INT32_MAX - kDN || r < kDK || r > DSPARK_DRAFT_MAX_RANK || r % kDK != 0 ||
      !(temperature > 0.0f) || !std::isfinite(temperature))
    return DSPARK_ERR_INVALID_ARG;
  if (B == 0) return DSPARK_OK;
  if (!base_logits || !w1 || !w2t || !anchors || !uniforms || !draft_logits || !draft_tokens ||
      !device_status || !workspace)
    return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(base_logits) || !aligned16(w1) || !aligned16(w2t) || !aligned16(draft_logits) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return DSPARK_ERR_INVALID_ARG;
  if (workspace_bytes < DSPARK_DRAFT_WS_BYTES(B, r, V)) return DSPARK_ERR_WORKSPACE;
  int sms = 0;
  bool coop = false;
  if (int rc = draft_setup(sms, coop)) return rc;

  const int Vi = static_cast<int>(V);
  const int n_tiles = (Vi + kDN - 1) / kDN;
  const int n_m = (B + kDM - 1) / kDM;
  int per_m = sms / n_m;
  if (per_m < 1) per_m = 1;
  if (per_m > n_tiles) per_m = n_tiles;
  uint16_t* G = static_cast<uint16_t*>(workspace);
  DraftStat* stats = reinterpret_cast<DraftStat*>(
      static_cast<char*>(workspace) + DSPARK_ALIGN256(static_cast<size_t>(B) * r * 2));
  DraftStat* stats1 = stats + DSPARK_ALIGN256(static_cast<size_t>(B) * n_tiles * 8) / 8;
  uint32_t* sync = reinterpret_cast<uint32_t*>(
      static_cast<char*>(workspace) + DSPARK_ALIGN256(static_cast<size_t>(B) * r * 2) +
      2 * DSPARK_ALIGN256(static_cast<size_t>(B) * n_tiles * 8));
  unsigned long long* ready =
      reinterpret_cast<unsigned long long*>(sync + 64);  // 256 bytes after the barrier words
  uint32_t* tile_sync = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(ready) +
                                                     DSPARK_ALIGN256(static_cast<size_t>(B) * 8 * kReadyStride));
  DraftPartial* parts =
      reinterpret_cast<DraftPartial*>(reinterpret_cast<char*>(tile_sync) + kTileSyncBytes);

  CUtensorMap mapW, mapU, mapL;
  {
    const cuuint64_t sg[1] = {static_cast<cuuint64_t>(r) * 2};
    const cuuint32_t bw[2] = {kDK, kDN};
    const cuuint64_t dw[2] = {static_cast<cuuint64_t>(r), static_cast<cuuint64_t>(V)};
    const cuuint64_t du[3] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(gamma),
                              static_cast<cuuint64_t>(B)};
    const cuuint64_t su[2] = {static_cast<cuuint64_t>(V) * 2,
                              static_cast<cuuint64_t>(V) * 2 * static_cast<cuuint64_t>(gamma)};
    const cuuint32_t bu[3] = {kDK, 1, kDM};
    if (!encode_map(&mapW, w2t, 2, dw, sg, bw) ||
        !encode_map(&mapU, base_logits, 3, du, su, bu) ||
        !encode_map(&mapL, draft_logits, 3, du, su, bu))
      return DSPARK_ERR_CUDA;
  }

  const ExpParams ep = draft_exp_params(temperature);
  const uint16_t* W1 = static_cast<const uint16_t*>(w1);
  if (ev && cudaEventRecord(ev[0], stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  const int grid = n_m * per_m;
  if (!ev && coop && n_m == 2 && sms > 2 * kPDrawCtas) {
    // two request tiles: the streaming CTAs serve both, and each tile's draws
    // (on kPDrawCtas CTAs of their own) and next G overlap the other tile's
    // streaming
    const int grid_all = sms < kMaxBlockCtas ? sms : kMaxBlockCtas;
    const int P = grid_all - kPDrawCtas < n_tiles ? grid_all - kPDrawCtas : n_tiles;
    if (cudaMemsetAsync(sync, 0,
                        256 + DSPARK_ALIGN256(static_cast<size_t>(B) * 8 * kReadyStride) + kTileSyncBytes,
                        stream) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    DraftBlockArgs ba{};
    ba.s = DraftStepArgs{B, Vi, r, gamma, 0, n_tiles, n_m, P, ep, stats, device_status};
    ba.p = DraftPickArgs{B,     Vi,       r, gamma, 0,  n_tiles, ep, stats,
                         static_cast<const uint16_t*>(draft_logits), uniforms, W1, G,
                         draft_tokens, device_status, nullptr};
    ba.k_begin = 0;
    ba.k_end = gamma;
    ba.G = nullptr;
    ba.stats1 = stats1;
    ba.anchors = anchors;
    ba.sync = sync;
    ba.ready = ready;
    ba.parts = parts;
    ba.tile_sync = tile_sync;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = P + kPDrawCtas;
    cfg.blockDim = kPThreads;
    cfg.dynamicSmemBytes = kPairSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_draft_pair, mapW, mapU, mapL, ba) == cudaSuccess)
      return DSPARK_OK;
    (void)cudaGetLastError();  // not resident as one grid: the other paths
  }
  if (!ev && coop && grid <= sms && grid <= kMaxBlockCtas) {
    // the whole block in one cooperative launch (every CTA resident, one per SM)
    if (cudaMemsetAsync(sync, 0,
                        256 + DSPARK_ALIGN256(static_cast<size_t>(B) * 8 * kReadyStride) + kTileSyncBytes,
                        stream) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    DraftBlockArgs ba{};
    ba.s = DraftStepArgs{B, Vi, r, gamma, 0, n_tiles, n_m, per_m, ep, stats, device_status};
    ba.p = DraftPickArgs{B,     Vi,       r, gamma, 0,  n_tiles, ep, stats,
                         static_cast<const uint16_t*>(draft_logits), uniforms, W1, G,
                         draft_tokens, device_status, nullptr};
    ba.k_begin = 0;
    ba.k_end = gamma;
    ba.G = nullptr;
    ba.stats1 = stats1;
    ba.anchors = anchors;
    ba.sync = sync;
    ba.ready = ready;
    ba.parts = parts;
    ba.tile_sync = tile_sync;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = kDThreads;
    cfg.dynamicSmemBytes = kDraftSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_draft_block, mapW, mapU, mapL, ba) == cudaSuccess)
      return DSPARK_OK;
    (void)cudaGetLastError();  // not resident as one grid: fall back to one launch per step
  }
  if (launch_plain(k_draft_gather, B, 32, 0, stream, anchors, W1, G, B, Vi, r, device_status) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (ev && cudaEventRecord(ev[1], stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  for (int k = 0; k < gamma; ++k) {
    DraftBlockArgs sa{};
    sa.s = DraftStepArgs{B, Vi, r, gamma, k, n_tiles, n_m, per_m, ep, stats, device_status};
    sa.p = DraftPickArgs{B,     Vi,       r, gamma, k,  n_tiles, ep, stats,
                         static_cast<const uint16_t*>(draft_logits), uniforms, W1, G,
                         draft_tokens, device_status, nullptr};
    sa.k_begin = k;
    sa.k_end = k + 1;
    sa.G = G;
    if (launch_plain(k_draft_step, n_m * per_m, kDThreads, kDraftSmem, stream, mapW, mapU, mapL,
                     sa) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    if (ev && cudaEventRecord(ev[2 + 2 * k], stream) != cudaSuccess) return DSPARK_ERR_CUDA;
    DraftPickArgs pa{B,     Vi,       r, gamma, k,  n_tiles, ep, stats,
                     static_cast<const uint16_t*>(draft_logits), uniforms, W1, G, draft_tokens,
                     device_status, nullptr};
    if (launch_plain(k_draft_pick, (B + kPickWarps - 1) / kPickWarps, kPickWarps * 32, 0, stream,
                     pa) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    if (ev && cudaEventRecord(ev[3 + 2 * k], stream) != cudaSuccess) return DSPARK_ERR_CUDA;
  }
  return DSPARK_OK;
}

}  // namespace
}  // namespace dspark

extern "C" int dspark_draft_markov(const void* base_logits, const void* w1, const void* w2t,
                                   const int32_t* anchors, const float* uniforms,
                                   float temperature, int32_t B, int32_t gamma, int64_t V,
                                   int32_t r, void* draft_logits, int32_t* draft_tokens,
                                   int32_t* device_status, void* workspace,
                                   size_t workspace_bytes, struct CUstream_st* stream) {
  return dspark::draft_entry(base_logits, w1, w2t, anchors, uniforms, temperature, B, gamma, V, r,
                             draft_logits, draft_tokens, device_status, workspace,
                             workspace_bytes, stream, nullptr);
}

extern "C" int dspark_draft_markov_timed(const void* base_logits, const void* w1, const void* w2t,
                                         const int32_t* anchors, const float* uniforms,
                                         float temperature, int32_t B, int32_t gamma, int64_t V,
                                         int32_t r, void* draft_logits, int32_t* draft_tokens,
                                         int32_t* device_status, void* workspace,
                                         size_t workspace_bytes, struct CUstream_st* stream,
                                         struct CUevent_st** events) {
  if (!events || gamma < 1 || gamma > DSPARK_MAX_GAMMA) return DSPARK_ERR_INVALID_ARG;
  for (int i = 0; i < 2 * gamma + 2; ++i)
    if (!events[i]) return DSPARK_ERR_INVALID_ARG;
  return dspark::draft_entry(base_logits, w1, w2t, anchors, uniforms, temperature, B, gamma, V, r,
                             draft_logits, draft_tokens, device_status, workspace,
                             workspace_bytes, stream, events);
}

// A diagnostic (no counterpart in the paper): one bounded wait that runs out.
extern "C" int dspark_wait_selftest(int32_t which, void* sync_words, int32_t* device_status,
                                    struct CUstream_st* stream) {
  if ((which != 0 && which != 1) || !device_status || (which == 1 && !sync_words) ||
      (reinterpret_cast<uintptr_t>(sync_words) & 7u) != 0)
    return DSPARK_ERR_INVALID_ARG;
  dspark::k_wait_selftest<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      which, static_cast<uint32_t*>(sync_words), device_status);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
