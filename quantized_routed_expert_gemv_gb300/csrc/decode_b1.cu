// decode_b1.cu -- single-token decode (B = 1), the latency-critical case.
//
// Same three steps as decode.cu (router + top-k + grouping, gate|up +
// SwiGLU, down + combine; TurboFieldfare page, section "Token üretim
// süreci"), with an inner loop built for one token:
//
// Integer dot products (the fixed-point path of gemv.cuh): every 32-value
// chunk of activations becomes 16-bit fixed point with its own power-of-two
// exponent and dp4a accumulates the chunk's code x activation products
// exactly; the affine bias term b * sum_j x_j is added in fp32.  Per 32
// codes this costs ~35 instructions instead of ~78 for unpack-to-float +
// FFMA, which keeps the CUDA cores well ahead of HBM.  The router keeps the
// float path: its top-k must agree with an fp64 evaluation to within a
// 1e-3 logit margin, and fp32 products of 8-bit codes and bf16 activations
// are exact.
//
// router_b1_kernel  8-bit router rows (float path); the last CTA takes the
//                   top-k with bitonic sorts and merges across its 16 warps
//                   on (logit, id) keys.
// ffn_b1_kernel     the step's gate|up and down work as one claimed item list
//                   in one persistent kernel (the layer's usual path): gate|up
//                   items publish fixed-point h groups, then down items copy
//                   the expert's h block with their weights, and per row tile
//                   the last expert's epilogue sums the experts' rows in a
//                   fixed order.
// The expert cache runs the same step as separate kernels, so the shared
// expert's gate|up can run while missing records are copied:
// gateup_b1_kernel  each consumer thread converts its chunk of the token's
//                   hidden state; items are streamed as in decode.cu.  An
//                   epilogue warp gathers each item's row sums, applies
//                   SwiGLU and writes the item's h values as fixed-point
//                   8-value groups, each with its own exponent, so consumer
//                   warps never meet at a barrier or wait on an epilogue.
// down_b1_kernel    copies each expert's fixed-point h block into a small
//                   ring ahead of its weight tiles and streams the CTA's row
//                   tiles expert by expert; partial sums stay in registers
//                   across experts (weighted by p_i), one reduction per tile.
#include <algorithm>
#include <cfloat>

#include "common.cuh"
#include "fused.cuh"
#include "gemv.cuh"
#include "kernels.h"

namespace moe {


// ============================================================================
// Router (B = 1): 8-bit rows against the fixed-point token, then top-k.
// ============================================================================

// ---- block-wide top-k ------------------------------------------------------
// A candidate is one 64-bit key: the logit's IEEE bits mapped to an
// order-preserving unsigned in the high word (every finite logit maps above
// 0), 0xFFFFFFFF - id in the low word, so a larger key is a larger logit and,
// on a tie, the lower id.  0 marks an absent candidate.
__device__ __forceinline__ uint64_t tk_key(float l, int e) {
  const uint32_t u = __float_as_uint(l + 0.0f);  // -0 and +0 compare equal: one key
  const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(k) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(e));
}

__device__ __forceinline__ float tk_logit(uint64_t key) {
  const uint32_t k = static_cast<uint32_t>(key >> 32);
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(kAll, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(kAll, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Bitonic sort of the warp's 32 keys, largest in lane 0.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
  for (int k2 = 2; k2 <= 32; k2 <<= 1)
#pragma unroll
    for (int j = k2 >> 1; j > 0; j >>= 1) {
      const uint64_t o = shfl_xor64(v, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k2) == 0);
      v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  return v;
}

// Top 32 of two descending lists held one key per lane (a) and (b), returned
// descending: max(a[i], b[31 - i]) is bitonic and holds the 32 largest; the
// half-cleaners sort it.
__device__ __forceinline__ uint64_t warp_merge_desc(uint64_t a, uint64_t b_rev, int lane) {
  uint64_t v = a > b_rev ? a : b_rev;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t o = shfl_xor64(v, j);
    v = ((lane & j) == 0) ? (v > o ? v : o) : (v < o ? v : o);
  }
  return v;
}

// Bitonic sort of the warp's 32 values, smallest in lane 0.
__device__ __forceinline__ uint32_t warp_sort_asc32(uint32_t v, int lane) {
#pragma unroll
  for (int k2 = 2; k2 <= 32; k2 <<= 1)
#pragma unroll
    for (int j = k2 >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(kAll, v, j);
      const bool keep_min = ((lane & j) == 0) == ((lane & k2) == 0);
      v = keep_min ? min(v, o) : max(v, o);
    }
  return v;
}

// Top-k of one token's E <= 1024 logits (logit(e) reads one) by the whole
// 16-warp block, then the softmax over the chosen logits and the
// single-token grouping.  Warp w sorts candidates 32w .. 32w + 31 (and, for
// E > 512, merges in 512 + 32w ..); a tree of warp merges halves the lists
// four times, so warp 0 ends with the 32 largest keys in order.  The result
// is the selection by (logit descending, id ascending), as the repeated
// argmax defines it.  `lists` is [16][32] keys of shared memory.
template <typename Logit>
__device__ __forceinline__ void topk_block_b1(const LayerArgs& a, uint64_t (*lists)[32], Logit logit) {
  const int E = a.E, k = a.k, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int e = warp * 32 + lane;
  uint64_t v = warp_sort_desc(e < E ? tk_key(logit(e), e) : 0ull, lane);
  e += 512;
  if (E > 512) {
    const uint64_t w2 = warp_sort_desc(e < E ? tk_key(logit(e), e) : 0ull, lane);
    v = warp_merge_desc(v, shfl_xor64(w2, 31), lane);
  }
  lists[warp][lane] = v;
  __syncthreads();
#pragma unroll
  for (int n = 8; n >= 1; n >>= 1) {
    if (warp < n) lists[warp][lane] = warp_merge_desc(lists[warp][lane], lists[warp + n][31 - lane], lane);
    __syncthreads();
  }
  if (warp != 0) return;
  const uint64_t key = lists[0][lane];
  int myi = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
  float myl = tk_logit(key);
  if (lane < k && (key == 0ull || myi >= E)) {  // only with non-finite logits (outside the contract)
    latch_error(&a.ws.ctl[0], kErrRange);
    myi = lane, myl = 0.f;
  }
  const float lmax = __shfl_sync(kAll, myl, 0);
  const float ex = (lane < k) ? expf(myl - lmax) : 0.f;
  const float z = warp_add(ex);
  if (lane < k) {
    a.ids[lane] = myi, a.weights[lane] = ex / z;
    if (a.ids_host) a.ids_host[lane] = myi, a.weights_host[lane] = ex / z;
  }
  // grouping for one token: active experts in ascending id, one pair each;
  // the sort carries each expert's position in ids[] in the low 5 bits
  const uint32_t s = warp_sort_asc32(lane < k ? (static_cast<uint32_t>(myi) << 5) | lane : 0xFFFFFFFFu, lane);
  if (lane < k) {
    a.ws.act_expert[lane] = static_cast<int>(s >> 5);
    a.ws.act_off[lane] = lane;
    a.ws.act_cnt[lane] = 1;
    a.ws.pair_token[lane] = 0;
    a.ws.pair_slot[lane] = static_cast<int>(s & 31u);
  }
  if (lane == 0) *a.ws.n_act = k;
}


constexpr int kR1Threads = 512;
constexpr int kR1Rows = 4;  // rows per CTA pass: 128 CTAs for 512 experts (the router's latency is on the critical path)

__global__ void __launch_bounds__(kR1Threads) router_b1_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(16) float rsm[];
  if (blockIdx.x == 0 && threadIdx.x == 0) a.ws.ctl[3] = 0u;  // shared-only gate|up claims
  const int H = a.H, E = a.E;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int NW = kR1Threads / 32;
  const int nchunk = H >> 4;  // 16 8-bit codes per chunk
  const bool act = tid < nchunk;
  float* red = rsm;  // [kR1Rows][NW]

  uint4 q[kR1Rows];
  uint32_t sbw[kR1Rows];
  auto load_rows = [&](int e0) {
#pragma unroll
    for (int r = 0; r < kR1Rows; ++r) {
      q[r] = make_uint4(0, 0, 0, 0), sbw[r] = 0;
      if (act && e0 + r < E) {
        q[r] = __ldg(reinterpret_cast<const uint4*>(a.rcodes + static_cast<size_t>(e0 + r) * H) + tid);
        sbw[r] = __ldg(a.rsb + static_cast<size_t>(e0 + r) * (H >> 6) + (tid >> 2));
      }
    }
  };
  load_rows(blockIdx.x * kR1Rows);  // weight rows in flight before the activations
  // When x is staged by the kernel before this one (x_pdl), wait for it; the
  // dependents (which read x too) are released only after that, so they see
  // x complete.  Launched in plain stream order, the wait returns at once.
  pdl_wait();
  pdl_launch_dependents();

  // token chunk: 16 bf16 activations, pre-scaled per byte position
  float2 X[8];
  float sx = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) X[j] = make_float2(0.f, 0.f);
  if (act) {
    const uint4* xp = reinterpret_cast<const uint4*>(a.x + tid * 16);
    const uint4 x0 = __ldg(xp), x1 = __ldg(xp + 1);
    const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float lo = bf16lo(xw[j]), hi = bf16hi(xw[j]);
      X[j] = make_float2(lo * byte_scale((2 * j) & 3), hi * byte_scale((2 * j + 1) & 3));
      sx += lo;
      sx += hi;
    }
  }

  for (int e0 = blockIdx.x * kR1Rows; e0 < E; e0 += gridDim.x * kR1Rows) {
    if (e0 != blockIdx.x * kR1Rows) load_rows(e0);
#pragma unroll
    for (int r = 0; r < kR1Rows; ++r) {
      const float p = fmaf(bf16lo(sbw[r]) * 0x1p64f, dot16_u8(q[r], X), bf16hi(sbw[r]) * sx);
      const float v = warp_add(p);
      if (lane == 0) red[r * NW + warp] = v;
    }
    __syncthreads();
    if (tid < kR1Rows && e0 + tid < E) {
      float v = 0.f;
      for (int w = 0; w < NW; ++w) v += red[tid * NW + w];
      a.ws.logits[e0 + tid] = v + (a.beta ? __ldg(a.beta + e0 + tid) : 0.f);
    }
    __syncthreads();
  }

  // ---- last CTA: top-k, weights, grouping (one token) ---------------------
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&a.ws.ctl[1], 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  __shared__ uint64_t lists[16][32];
  topk_block_b1(a, lists, [&](int e) { return __ldcg(a.ws.logits + e); });
  if (tid == 0) a.ws.ctl[1] = 0u;
}

size_t router_b1_smem_bytes(int E) {
  return std::max(static_cast<size_t>(kR1Rows) * (kR1Threads / 32) * 4, static_cast<size_t>(E) * 4);
}

// ============================================================================
// gate|up + SwiGLU (B = 1).  Consumer warp w: row-lane rl = w / WC owns
// gate rows 2rl, 2rl+1 and up rows 2rl, 2rl+1 of the item and column
// 32*(w % WC) + lane.  An item holds rth = 2*NRL gate rows and the same up
// rows of one expert (32 KB at H = 7168, so six stages fit); the shared
// expert's items come first.
// ============================================================================

constexpr int kG1Warps = 16;

constexpr int kG1Threads = (kG1Warps + 2) * 32;  // consumers, producer, epilogue warp

struct G1Smem {  // byte offsets of the dynamic shared-memory carve
  int wsum, item, bars, total;
};

__host__ __device__ inline G1Smem g1_smem(int nst, int stage, int rows) {
  G1Smem s;
  s.wsum = nst * stage;
  s.item = s.wsum + nst * kG1Warps * rows * 4;  // [NST] item index held by the stage
  s.bars = s.item + 64;
  s.total = s.bars + 3 * nst * 8 + 16;          // full, empty, partial sums done
  return s;
}


template <int R>  // rows per thread per item: R/2 gate + R/2 up
__global__ void __launch_bounds__(kG1Threads, 1) gateup_b1_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NCW = kG1Warps;
  const int H = a.H, C = H >> 5, WC = (C + 31) >> 5, NRL = a.gu_nrl, NAW = NRL * WC;
  constexpr int RH = R / 2;
  const int rth = RH * NRL;
  const int NST = a.gu_nst, SB = a.gu_stage;
  const G1Smem L = g1_smem(NST, SB, R);
  float* wsum = reinterpret_cast<float*>(smem + L.wsum);  // [NST][NCW][R]
  volatile int* s_item = reinterpret_cast<volatile int*>(smem + L.item);  // [NST]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + NST;  // consumers and the epilogue warp are done with a stage
  uint64_t* pdone = empty + NST;  // every consumer's partial sums of the stage's item are in
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&full[s], 1), mbar_init(&empty[s], NAW + 1), mbar_init(&pdone[s], NAW);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_launch_dependents();

  const int has_sh = a.Fs > 0 ? 1 : 0;
  const int tiles_s = has_sh ? a.Fs / rth : 0, tiles_r = a.F / rth;
  // Items 0 .. tiles_s-1: shared expert tiles (no routing needed).  Later
  // items need the router's output.  CTAs claim items from a global counter,
  // so CTAs that start late (their SM still ran the router) simply take fewer.

  if (warp == NCW) {  // ---------------- producer warp
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      // part 1 (shared expert only) counts its claims in ctl[3], which the
      // router of the next step clears; parts 0 and 2 in ctl[2], cleared by
      // the down kernel.  Part 2 starts after the shared items.
      const int part = a.gu_part;
      unsigned* claim = &a.ws.ctl[part == 1 ? 3 : 2];
      const int base = part == 2 ? tiles_s : 0;
      int it = 0, n_items = tiles_s;
      bool waited = false, marker = false;
      RingPos pos;
      int next = base + static_cast<int>(atomicAdd(claim, 1u));
      for (;; ++it, pos.next(NST)) {
        const int i = next;
        if (i >= tiles_s && !waited && part != 1) {
          pdl_wait();
          waited = true;
          n_items = tiles_s + clamp_n_act(a) * tiles_r;
        }
        const int s = pos.s;
        if (it >= NST && !mbar_wait(&empty[s], pos.ph ^ 1u)) {
          latch_error(&a.ws.ctl[0], kErrTimeout);
          break;
        }
        if (i >= n_items) {  // no work left: tell the consumers through the ring
          s_item[s] = -1;
          mbar_arrive(&full[s]);
          marker = true;
          break;
        }
        next = base + static_cast<int>(atomicAdd(claim, 1u));  // claim ahead, latency overlaps the copy
        const int idx = i < tiles_s ? 0 : has_sh + (i - tiles_s) / tiles_r;
        const int tile = i < tiles_s ? i : (i - tiles_s) % tiles_r;
        const B1Entry en = b1_entry(a, idx, has_sh);
        if (!en.shared && a.slot_tag && a.slot_tag[en.slot] != en.expert)
          latch_error(&a.ws.ctl[0], kErrResidency);
        const size_t j0 = static_cast<size_t>(tile) * rth;
        const uint32_t cb = rth * (H / 2), sbb = rth * (H / 16);
        uint8_t* st = smem + s * SB;
        s_item[s] = i;
        mbar_arrive_expect_tx(&full[s], 2 * cb + 2 * sbb);
        bulk_g2s(st, en.rec + en.off->gate_codes + j0 * (H / 2), cb, &full[s], pol);
        bulk_g2s(st + cb, en.rec + en.off->up_codes + j0 * (H / 2), cb, &full[s], pol);
        bulk_g2s(st + 2 * cb, en.rec + en.off->gate_sb + j0 * (H / 16), sbb, &full[s], pol);
        bulk_g2s(st + 2 * cb + sbb, en.rec + en.off->up_sb + j0 * (H / 16), sbb, &full[s], pol);
      }
      // Copies in flight land before exit.  The end marker re-armed the stage
      // of item it - NST, whose copies were already consumed (its empty wait
      // passed), so that one is skipped: its parity would alias.
      for (int j = max(0, it - NST + (marker ? 1 : 0)); j < it; ++j)
        if (!mbar_wait(&full[j % NST], (j / NST) & 1)) latch_error(&a.ws.ctl[0], kErrTimeout);
    }
    return;
  }

  if (warp == NCW + 1) {  // ---------------- epilogue warp
    // Per item, in ring order: gather the gate and up sums of the item's
    // rows (at most 64: two per lane), release the stage, then SwiGLU and
    // the fixed-point h groups, off the consumers' path.
    RingPos pos;
    for (;; pos.next(NST)) {
      const int s = pos.s;
      if (!mbar_wait_sleep_warp(&full[s], pos.ph)) {
        if (lane == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
        break;
      }
      const int i = s_item[s];
      if (i < 0) break;  // the producer ran out of items
      if (!mbar_wait_sleep_warp(&pdone[s], pos.ph)) {
        if (lane == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
        break;
      }
      float gs[2] = {0.f, 0.f}, us[2] = {0.f, 0.f};
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int j = q * 32 + lane;
        if (j < rth) {
          const int rlj = j / RH, mj = j % RH;
          for (int w = 0; w < WC; ++w) {
            const float* ws = wsum + (s * NCW + rlj * WC + w) * R;
            gs[q] += ws[mj];
            us[q] += ws[RH + mj];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      // entry idx of the step (shared expert first, then the active experts
      // in ascending id) owns h chunks c0 .. c0 + nc - 1; the item's rth
      // rows (a multiple of 8) are whole groups
      const int idx = i < tiles_s ? 0 : has_sh + (i - tiles_s) / tiles_r;
      const int tile = i < tiles_s ? i : (i - tiles_s) % tiles_r;
      const bool sh_row = has_sh && idx == 0;
      const int nc = (sh_row ? a.Fs : a.F) >> 5;
      const int c0 = sh_row ? 0 : has_sh * (a.Fs >> 5) + (idx - has_sh) * (a.F >> 5);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int j = q * 32 + lane;
        if (q * 32 < rth) publish_hgroup(a, c0, nc, tile * rth + j, silu1(gs[q]) * us[q], j < rth, lane);
      }
    }
    return;
  }

  // ---------------------------------------------------- consumers
  const int rl = warp / WC, wc = warp % WC, col = wc * 32 + lane;
  const bool has_col = col < C;
  if (warp >= NAW) return;  // no column of this item layout
  float xv[32], sx = 0.f;
#pragma unroll
  for (int m = 0; m < 32; ++m) xv[m] = 0.f;
  if (has_col) {
    const uint4* v = reinterpret_cast<const uint4*>(a.x + col * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 t = __ldg(v + i);
      const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) xv[8 * i + 2 * j] = bf16lo(w4[j]), xv[8 * i + 2 * j + 1] = bf16hi(w4[j]);
    }
#pragma unroll
    for (int m = 0; m < 32; ++m) sx += xv[m];
  }
  XChunk X;
  const float scale = make_xchunk_own(xv, X);

  RingPos pos;
  for (;; pos.next(NST)) {
    const int s = pos.s;
    if (!mbar_wait_sleep_warp(&full[s], pos.ph)) {
      if (lane == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
      break;
    }
    const int i = s_item[s];
    if (i < 0) break;  // the producer ran out of items
    const uint8_t* st = smem + s * SB;
    const uint8_t* stsb = st + 2 * rth * (H / 2);
    float part[R];
#pragma unroll
    for (int m = 0; m < R; ++m) part[m] = 0.f;
    if (has_col) {
#pragma unroll
      for (int m = 0; m < R; ++m) {
        const int r = (m < RH) ? (RH * rl + m) : (rth + RH * rl + m - RH);
        const uint4 q = *reinterpret_cast<const uint4*>(st + r * (H / 2) + col * 16);
        const uint32_t sbw = *reinterpret_cast<const uint32_t*>(stsb + r * (H / 16) + (col >> 1) * 4);
        part[m] = fmaf(bf16lo(sbw) * scale, static_cast<float>(dot_chunk(q, X)), bf16hi(sbw) * sx);
      }
    }
    constexpr int LPR = 32 / R;  // lanes per row after the butterfly
    float v;
    if constexpr (R == 8) v = bfly8(part, lane);
    else v = bfly4b(part, lane);
    if ((lane & (LPR - 1)) == 0) wsum[(s * NCW + warp) * R + lane / LPR] = v;
    __syncwarp();  // the lanes' sums before lane 0's arrivals (release at CTA scope)
    if (lane == 0) mbar_arrive(&pdone[s]), mbar_arrive(&empty[s]);
  }
  pdl_wait();  // the grid completes after the router's, which the down kernel relies on
}

size_t gateup_b1_smem_bytes(const LayerArgs& a, int rows) {
  return g1_smem(a.gu_nst, a.gu_stage, rows).total;
}

// ============================================================================
// down + combine (B = 1).  Prologue: the producer streams the shared
// expert's first tiles before the dependency on gate|up (its weights need no
// routing); then a table of the step's experts (shared expert first, then
// active experts in ascending id: record, width, fixed-point h chunks,
// routing weight).  Each expert's fixed-point h block (written by gate|up, a
// few KB) is bulk-copied into a small ring of its own ahead of the expert's
// weight tiles, so the weight ring gets nearly all of shared memory.  Main
// loop: experts outer, this CTA's row tiles of H inner (at most
// kD1MaxTiles), so a thread loads its activation chunk once per expert.  A
// thread owns column `col` and rows rl + NRL*m (m < 2) of every tile for
// each expert width; the weighted sums stay in registers until the end,
// when one butterfly + one barrier per CTA combine them.
// ============================================================================

constexpr int kD1MaxTiles = 4;  // row tiles per CTA
constexpr int kD1Rpt = 2;       // rows per thread per tile and expert width
constexpr int kD1XSlots = 3;    // fixed-point h blocks in flight
constexpr int kD1MaxStages = 16;

struct D1Entry {        // one expert of the step, as the down kernel uses it
  const uint8_t* rec;   // record base
  float p;              // routing weight (1 for the shared expert)
  int Fe;               // FFN width
  int c0;               // first fixed-point chunk of its h row
  int expert;           // expert id (-1: shared)
};

struct D1Smem {
  int ent, xring, xslot, wsum, bars, total;
};

// rows: h rows of the step; ncmax: chunks of the widest h row.  An h slot
// holds one expert's h block: [4 kinds][nc] uint4 words, then nc float4
// group scales at 64 * nc, then nc float4 group sums at 80 * nc.
__host__ __device__ inline D1Smem d1_smem(int nst, int stage, int rows, int ncmax) {
  D1Smem s;
  s.ent = nst * stage;
  s.xring = s.ent + ((rows * static_cast<int>(sizeof(D1Entry)) + 127) / 128) * 128;
  s.xslot = (96 * ncmax + 127) / 128 * 128;
  s.wsum = s.xring + kD1XSlots * s.xslot;
  s.bars = s.wsum + kD1MaxTiles * kD1Warps * 4 * 4;  // [tile][warp][4]
  s.total = s.bars + (2 * nst + 2 * kD1XSlots) * 8 + 16;  // full, empty, h full, h empty
  return s;
}


__global__ void __launch_bounds__((kD1Warps + 1) * 32, 1) down_b1_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NCW = kD1Warps, NCT = NCW * 32, NX = kD1XSlots;
  const int RT = a.dn_rt, NST = a.dn_nst, SB = a.dn_stage, k = a.k;
  const int has_sh = a.Fs > 0 ? 1 : 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int max_rows = k + has_sh;
  const int ncmax = max(a.F, a.Fs) >> 5;
  const D1Smem L = d1_smem(NST, SB, max_rows, ncmax);
  D1Entry* ent = reinterpret_cast<D1Entry*>(smem + L.ent);
  uint8_t* xring = smem + L.xring;
  float* wsum = reinterpret_cast<float*>(smem + L.wsum);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + NST;
  uint64_t* xfull = empty + NST;  // fixed-point h block of an expert landed
  uint64_t* xempty = xfull + NX;  // ... and read by every consumer warp

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&full[s], 1), mbar_init(&empty[s], NCW);
    for (int s = 0; s < NX; ++s) mbar_init(&xfull[s], 1), mbar_init(&xempty[s], NCW);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_launch_dependents();
  // this CTA's tiles: blockIdx.x + t * gridDim.x, t < ntc (<= kD1MaxTiles by plan)
  const int n_tiles = a.dn_tiles;
  const int ntc = blockIdx.x < n_tiles ? min(kD1MaxTiles, (n_tiles - 1 - blockIdx.x) / gridDim.x + 1) : 0;
  const uint64_t pol = policy_evict_first();
  // the shared expert's tiles (entry 0) go out before the dependency wait
  const int pre = has_sh ? min(ntc, NST) : 0;
  if (warp == NCW && lane == 0) {
    const uint32_t cb = RT * (a.Fs / 2), sbb = RT * (a.Fs / 16);
    for (int t = 0; t < pre; ++t) {
      const size_t r0 = static_cast<size_t>(blockIdx.x + t * gridDim.x) * RT;
      uint8_t* st = smem + t * SB;
      mbar_arrive_expect_tx(&full[t], cb + sbb);
      bulk_g2s(st, a.shared + a.off_s.down_codes + r0 * (a.Fs / 2), cb, &full[t], pol);
      bulk_g2s(st + cb, a.shared + a.off_s.down_sb + r0 * (a.Fs / 16), sbb, &full[t], pol);
    }
  }
  pdl_wait();  // fixed-point h, routing and weights are ready past this point
  if (blockIdx.x == 0 && tid == 0) a.ws.ctl[2] = 0u;  // gate|up claims: back to zero
  const int n_ent = min(clamp_n_act(a) + has_sh, max_rows);
  if (warp == 0) {
    for (int j = lane; j < n_ent; j += 32) {
      const B1Entry en = b1_entry(a, j, has_sh);
      D1Entry d;
      d.rec = en.rec;
      d.Fe = en.Fe;
      d.expert = en.expert;
      d.p = en.shared ? 1.f : a.weights[a.ws.pair_slot[en.pair]];
      d.c0 = en.shared ? 0 : has_sh * (a.Fs / 32) + (j - has_sh) * (a.F / 32);
      ent[j] = d;
      if (!en.shared && a.slot_tag && a.slot_tag[en.slot] != en.expert)
        latch_error(&a.ws.ctl[0], kErrResidency);
    }
  }
  __syncthreads();

  if (warp == NCW) {  // ---------------- producer warp: h blocks and expert weights
    if (lane == 0) {
      // the h words were written by the gate|up grid through the generic
      // proxy; the bulk copies read them through the async proxy
      asm volatile("fence.proxy.async.global;" ::: "memory");
      int it = 0, jx = 0;
      bool stop = false;
      RingPos pos;
      for (int j = 0; j < n_ent && !stop; ++j) {
        const D1Entry d = ent[j];
        const int xs = j % NX, nc = d.Fe / 32;
        if (j >= NX && !mbar_wait(&xempty[xs], ((j / NX) & 1) ^ 1u)) {
          latch_error(&a.ws.ctl[0], kErrTimeout);
          break;
        }
        uint8_t* xb = xring + xs * L.xslot;
        mbar_arrive_expect_tx(&xfull[xs], 96 * nc);
        // every CTA reads these blocks: no evict-first hint
        bulk_g2s(xb, a.ws.hx + static_cast<size_t>(d.c0) * 96, 96 * nc, &xfull[xs]);
        jx = j + 1;
        const RecordOffsets& off = d.expert < 0 ? a.off_s : a.off_r;
        const uint32_t cb = RT * (d.Fe / 2), sbb = RT * (d.Fe / 16);
        for (int t = 0; t < ntc; ++t, ++it, pos.next(NST)) {
          if (j == 0 && t < pre) continue;  // issued before the dependency wait
          const int s = pos.s;
          if (it >= NST && !mbar_wait(&empty[s], pos.ph ^ 1u)) {
            latch_error(&a.ws.ctl[0], kErrTimeout);
            stop = true;
            break;
          }
          const size_t r0 = static_cast<size_t>(blockIdx.x + t * gridDim.x) * RT;
          uint8_t* st = smem + s * SB;
          mbar_arrive_expect_tx(&full[s], cb + sbb);
          bulk_g2s(st, d.rec + off.down_codes + r0 * (d.Fe / 2), cb, &full[s], pol);
          bulk_g2s(st + cb, d.rec + off.down_sb + r0 * (d.Fe / 16), sbb, &full[s], pol);
        }
      }
      // copies in flight land before exit
      for (int j = max(0, it - NST); j < it; ++j)
        if (!mbar_wait(&full[j % NST], (j / NST) & 1)) latch_error(&a.ws.ctl[0], kErrTimeout);
      for (int j = max(0, jx - NX); j < jx; ++j)
        if (!mbar_wait(&xfull[j % NX], (j / NX) & 1)) latch_error(&a.ws.ctl[0], kErrTimeout);
    }
    return;
  }

  // ---- main loop (consumer warps): experts outer, tiles inner
  const D1Geo gs = d1_geo(has_sh ? a.Fs : a.F, warp, lane), gr = d1_geo(a.F, warp, lane);
  float acc[kD1MaxTiles][2 * kD1Rpt];  // [tile][shared rows m, routed rows m]
#pragma unroll
  for (int t = 0; t < kD1MaxTiles; ++t)
#pragma unroll
    for (int m = 0; m < 2 * kD1Rpt; ++m) acc[t][m] = 0.f;
  bool abort = false;  // this warp gave up a wait; acted on at the final barrier
  RingPos pos;
  for (int j = 0; j < n_ent; ++j) {
    const D1Entry d = ent[j];
    const bool sh = d.expert < 0;
    const D1Geo& g = sh ? gs : gr;
    XChunk X;
    float scp[4] = {0.f, 0.f, 0.f, 0.f}, psx = 0.f;
    const int xs = j % NX;
    if (!abort && !mbar_wait_sleep_warp(&xfull[xs], (j / NX) & 1)) {
      if (lane == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
      abort = true;
    }
    if (!abort && g.act) {
      const int C = g.C, col = g.col;
      const uint8_t* xb = xring + xs * L.xslot;
      const uint4* xw = reinterpret_cast<const uint4*>(xb);
      const uint4 g0 = xw[0 * C + col], g1 = xw[1 * C + col], g2 = xw[2 * C + col], g3 = xw[3 * C + col];
      X.eh[0] = g0.x, X.eh[1] = g0.y, X.eh[2] = g0.z, X.eh[3] = g0.w;
      X.el[0] = g1.x, X.el[1] = g1.y, X.el[2] = g1.z, X.el[3] = g1.w;
      X.oh[0] = g2.x, X.oh[1] = g2.y, X.oh[2] = g2.z, X.oh[3] = g2.w;
      X.ol[0] = g3.x, X.ol[1] = g3.y, X.ol[2] = g3.z, X.ol[3] = g3.w;
      const float4 sc4 = reinterpret_cast<const float4*>(xb + 64 * C)[col];
      const float4 sm4 = reinterpret_cast<const float4*>(xb + 80 * C)[col];
      scp[0] = sc4.x * d.p, scp[1] = sc4.y * d.p, scp[2] = sc4.z * d.p, scp[3] = sc4.w * d.p;
      psx = d.p * ((sm4.x + sm4.y) + (sm4.z + sm4.w));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&xempty[xs]);
    const int rowb = (d.Fe / 2), sbrow = (d.Fe / 16);
#pragma unroll
    for (int t = 0; t < kD1MaxTiles; ++t) {
      if (t >= ntc) break;
      const int s = pos.s;
      const uint32_t ph = pos.ph;
      pos.next(NST);
      if (abort) continue;
      if (!mbar_wait_sleep_warp(&full[s], ph)) {
        if (lane == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
        abort = true;
        continue;
      }
      if (g.act) {
        const uint8_t* st = smem + s * SB;
        const uint8_t* stsb = st + RT * rowb;
#pragma unroll
        for (int m = 0; m < kD1Rpt; ++m) {
          const int r = g.rl + g.NRL * m;
          if (r < RT) {
            const uint4 q = *reinterpret_cast<const uint4*>(st + r * rowb + g.col * 16);
            const uint32_t sbw = *reinterpret_cast<const uint32_t*>(stsb + r * sbrow + (g.col >> 1) * 4);
            const float v = fmaf(bf16lo(sbw), dot_chunk_g(q, X, scp), bf16hi(sbw) * psx);
            if (sh) acc[t][m] += v;
            else acc[t][kD1Rpt + m] += v;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  // ---- combine: per tile, one butterfly; one barrier for the whole CTA
#pragma unroll
  for (int t = 0; t < kD1MaxTiles; ++t) {
    if (t >= ntc) break;
    const float v = bfly4b(acc[t], lane);  // lane L: value (L >> 3) = [sh m0, sh m1, rt m0, rt m1]
    if ((lane & 7) == 0) wsum[(t * NCW + warp) * 4 + (lane >> 3)] = v;
  }
  if (named_bar_or(1, NCT, abort)) return;  // uniform exit if any warp gave up
  for (int q = tid; q < ntc * RT; q += NCT) {
    const int t = q / RT, r = q % RT;
    float out = 0.f;
    if (has_sh) {
      const int rl = r % gs.NRL, m = r / gs.NRL;
      for (int w = 0; w < gs.WC; ++w) out += wsum[(t * NCW + rl * gs.WC + w) * 4 + m];
    }
    {
      const int rl = r % gr.NRL, m = r / gr.NRL;
      for (int w = 0; w < gr.WC; ++w) out += wsum[(t * NCW + rl * gr.WC + w) * 4 + kD1Rpt + m];
    }
    const size_t o = static_cast<size_t>(blockIdx.x + t * gridDim.x) * RT + r;
    a.out_bf16[o] = f32_to_bf16_rne(out);
    if (a.out_f32) a.out_f32[o] = out;
  }
}

size_t down_b1_smem_bytes(const LayerArgs& a) {
  const int has_sh = a.Fs > 0 ? 1 : 0;
  return d1_smem(a.dn_nst, a.dn_stage, a.k + has_sh, std::max(a.F, a.Fs) / 32).total;
}

// ============================================================================
// Fused gate|up + down (B = 1): one persistent kernel, one HBM stream.
//
// The step's work is one list of items claimed from a global counter: gate|up
// items (rth gate + rth up rows of one expert, as in gateup_b1_kernel) and
// down items (RTD rows of H of one expert's down matrix, with the expert's
// fixed-point h block copied in the same stage).  The list runs
//   G(0) ... G(n - 1) D(0) ... D(n - 1)
// (entry 0 the shared expert): every gate|up item, then every down item, so
// a CTA reaches an expert's down items long after that expert's last
// gate|up item was claimed and its h is complete; the producer still checks
// a per-expert completion counter before it issues a down item.  The stream
// never stops at a kernel boundary between the two halves.
//
// Warps: NCW consumers, one producer, two epilogue warps that take ring
// positions in turn.  For a gate|up item the epilogue applies SwiGLU and
// writes the fixed-point h groups, then counts the item for its expert
// (release).  For a down item it writes the item's weighted row sums to
// ypart[expert] and counts the expert for the row tile (acquire-release);
// the epilogue that completes a tile sums its rows over the experts in
// entry order (the same order whichever CTAs did the work) and writes the
// output.  Every counter is back at zero when the step ends: the row-tile
// counters by the tile's summing epilogue, the claim and per-expert counters
// by the last producer to finish claiming.
// ============================================================================

constexpr int kF1Warps = 16;                     // consumer warps
constexpr int kF1Threads = (kF1Warps + 3) * 32;  // + producer + two epilogue warps
constexpr int kF1SmemBudget = 222 * 1024;
constexpr int kF1MaxStages = 16;

struct F1Smem {
  int wsum, info, ent, bars, total;
};

struct F1Ent {          // one expert of the step, as the fused producer uses it
  const uint8_t* rec;   // record base
  float p;              // routing weight (1 for the shared expert)
  int c0;               // first fixed-point chunk of its h row
  unsigned need;        // gate|up items that complete its h
  int pad;
};

__host__ __device__ inline F1Smem f1_smem(int nst, int stage) {
  F1Smem s;
  s.wsum = nst * stage;                      // [NST][NCW][8] per-warp row sums
  s.info = s.wsum + nst * kF1Warps * 8 * 4;  // [16] item codes, [16] routing weights
  s.ent = s.info + 2 * kF1MaxStages * 4 + 16;  // (+16: the step's expert count) expert table
  s.bars = s.ent + (kMaxTopK + 1) * static_cast<int>(sizeof(F1Ent));
  s.total = s.bars + 3 * nst * 8 + 16;       // full, empty, partial sums done
  return s;
}


template <int R>  // gate|up rows per thread per item: R/2 gate + R/2 up
__global__ void __launch_bounds__(kF1Threads, 1) ffn_b1_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NCW = kF1Warps;
  const int H = a.H, C = H >> 5, WC = (C + 31) >> 5, NRL = a.gu_nrl, NAW = NRL * WC;
  constexpr int RH = R / 2;
  const int rth = RH * NRL;
  const int NST = a.f1_nst, SB = a.f1_stage, RTD = a.f1_rt;
  const F1Smem L = f1_smem(NST, SB);
  float* wsum = reinterpret_cast<float*>(smem + L.wsum);
  volatile int* s_code = reinterpret_cast<volatile int*>(smem + L.info);
  volatile float* s_p = reinterpret_cast<volatile float*>(smem + L.info + kF1MaxStages * 4);
  volatile int* s_nent = reinterpret_cast<volatile int*>(smem + L.info + 2 * kF1MaxStages * 4);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + NST;   // consumers and the position's epilogue warp are done
  uint64_t* pdone = empty + NST;  // every consumer's row sums of the position are in
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&full[s], 1), mbar_init(&empty[s], NCW + 1), mbar_init(&pdone[s], NCW);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int has_sh = a.Fs > 0 ? 1 : 0;
  const int tiles_s = has_sh ? a.Fs / rth : 0, tiles_r = a.F / rth, ndn = H / RTD;
  const int n_pre = has_sh ? tiles_s : 0;  // items that need no routing: the shared gate|up

  if (warp == NCW) {  // ---------------- producer warp (lane 0 issues; the warp builds the table)
    F1Ent* tab = reinterpret_cast<F1Ent*>(smem + L.ent);
    const uint64_t pol = policy_evict_first(), pol_h = policy_evict_last();
    unsigned* claim = &a.ws.ctl[2];
    const F1Div dr = f1_div(tiles_r), dn = f1_div(ndn);
    int it = 0, n_items = n_pre, n_ent = has_sh, checked = -1, cur = 0, nxt = 0;
    bool ok = true;
    RingPos pos;
    if (has_sh && lane == 0) {  // the shared expert needs no routing
      F1Ent t;
      t.rec = a.shared, t.p = 1.f, t.c0 = 0, t.need = tiles_s;
      tab[0] = t;
    }
    if (lane == 0) {
      // claims run two items ahead, so a claim's round trip has a whole
      // item to complete before its index is needed
      cur = static_cast<int>(atomicAdd(claim, 1u));
      nxt = static_cast<int>(atomicAdd(claim, 1u));
    }
    for (int phase = 0; phase < 2 && ok; ++phase) {
      if (phase == 1) {
        // routed items: wait for the router, then the whole warp looks the
        // step's experts up once (lane j: routed expert j) into shared memory
        pdl_wait();
        const int n_act = clamp_n_act(a);
        for (int j = lane; j < n_act; j += 32) {
          const B1Entry en = b1_entry(a, has_sh + j, has_sh);
          if (a.slot_tag && a.slot_tag[en.slot] != en.expert) latch_error(&a.ws.ctl[0], kErrResidency);
          F1Ent t;
          t.rec = en.rec, t.p = a.weights[a.ws.pair_slot[en.pair]], t.c0 = has_sh * (a.Fs / 32) + j * (a.F / 32);
          t.need = tiles_r;
          tab[has_sh + j] = t;
        }
        __syncwarp();
        n_items = n_pre + n_act * tiles_r + (has_sh + n_act) * ndn;
        n_ent = has_sh + n_act;
        if (lane == 0) *s_nent = n_ent;  // for the epilogue warps, before any routed item is issued
      }
      if (lane == 0) {
        for (;; ++it, pos.next(NST)) {
          const int i = cur;
          if (phase == 0 && i >= n_pre) break;  // routed from here on: phase 1
          if (i >= n_items) break;
          cur = nxt;
          nxt = static_cast<int>(atomicAdd(claim, 1u));
          const int code = f1_item(i, has_sh, tiles_s, n_ent, dr, dn);
          const int gate = code & 1, e = code >> 20, tile = (code >> 1) & 0x7FFFF;
          const bool sh = has_sh && e == 0;
          const RecordOffsets& off = sh ? a.off_s : a.off_r;
          const F1Ent t = tab[e];
          // the completion check goes before the wait for a free stage, so
          // its latency overlaps it
          if (!gate && e != checked) {  // the expert's h must be complete before its block is copied
            if (!wait_count(&a.ws.hcnt[e], t.need)) {
              latch_error(&a.ws.ctl[0], kErrTimeout);
              ok = false;
              break;
            }
            checked = e;
            // h was written through the generic proxy; the bulk copy reads it
            // through the async proxy
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
          const int s = pos.s;
          if (it >= NST && !mbar_wait(&empty[s], pos.ph ^ 1u)) {
            latch_error(&a.ws.ctl[0], kErrTimeout);
            ok = false;
            break;
          }
          uint8_t* st = smem + s * SB;
          s_code[s] = code;
          if (gate) {
            const size_t j0 = static_cast<size_t>(tile) * rth;
            const uint32_t cb = rth * (H / 2), sbb = rth * (H / 16);
            mbar_arrive_expect_tx(&full[s], 2 * cb + 2 * sbb);
            bulk_g2s(st, t.rec + off.gate_codes + j0 * (H / 2), cb, &full[s], pol);
            bulk_g2s(st + cb, t.rec + off.up_codes + j0 * (H / 2), cb, &full[s], pol);
            bulk_g2s(st + 2 * cb, t.rec + off.gate_sb + j0 * (H / 16), sbb, &full[s], pol);
            bulk_g2s(st + 2 * cb + sbb, t.rec + off.up_sb + j0 * (H / 16), sbb, &full[s], pol);
          } else {
            const int Fe = sh ? a.Fs : a.F, nc = Fe / 32;
            const uint32_t cb = RTD * (Fe / 2), sbb = RTD * (Fe / 16), xb = 96 * nc;
            const size_t r0 = static_cast<size_t>(tile) * RTD;
            s_p[s] = t.p;
            mbar_arrive_expect_tx(&full[s], cb + sbb + xb);
            bulk_g2s(st, t.rec + off.down_codes + r0 * (Fe / 2), cb, &full[s], pol);
            bulk_g2s(st + cb, t.rec + off.down_sb + r0 * (Fe / 16), sbb, &full[s], pol);
            // the expert's h block, which every CTA reads: kept in L2
            bulk_g2s(st + cb + sbb, a.ws.hx + static_cast<size_t>(t.c0) * 96, xb, &full[s], pol_h);
          }
        }
      }
      ok = __shfl_sync(kAll, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0) {
      // copies in flight land before the end markers re-arm their stages
      for (int j = max(0, it - NST); j < it; ++j)
        if (!mbar_wait(&full[j % NST], (j / NST) & 1)) latch_error(&a.ws.ctl[0], kErrTimeout), ok = false;
      // one end marker per epilogue warp (positions it, it + 1); consumers
      // stop at the first
      for (int m = 0; m < 2; ++m, ++it, pos.next(NST)) {
        const int s = pos.s;
        if (it >= NST && !mbar_wait(&empty[s], pos.ph ^ 1u)) {
          latch_error(&a.ws.ctl[0], kErrTimeout);
          ok = false;
          break;
        }
        s_code[s] = -1;
        mbar_arrive(&full[s]);
      }
      // The last producer to get here resets the claim and per-expert
      // counters: every claim of the step is made and every down item's
      // completion check has passed, so every gate|up count is final.
      if (ok) {
        __threadfence();
        if (atomicAdd(&a.ws.ctl[8], 1u) == gridDim.x - 1) {
          a.ws.ctl[2] = 0u;
          for (int j = 0; j < n_ent; ++j) a.ws.hcnt[j] = 0u;
          a.ws.ctl[8] = 0u;
          __threadfence();
        }
      }
    }
    return;
  }

  if (warp > NCW) {  // ---------------- epilogue warps: ring positions q, q + 2, ...
    const int q = warp - NCW - 1;
    const D1Geo gs = d1_geo(has_sh ? a.Fs : a.F, 0, 0), gr = d1_geo(a.F, 0, 0);
    int n_ent = -1;  // known once the router's output is needed
    for (int it = q;; it += 2) {
      const int s = it % NST;
      const uint32_t ph = (it / NST) & 1;
      if (!mbar_wait_sleep_warp(&full[s], ph)) {
        if (lane == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
        break;
      }
      const int code = s_code[s];
      if (code < 0) break;
      if (!mbar_wait_sleep_warp(&pdone[s], ph)) {
        if (lane == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
        break;
      }
      const int gate = code & 1, e = code >> 20, tile = (code >> 1) & 0x7FFFF;
      const bool sh_row = has_sh && e == 0;
      float v0 = 0.f, v1 = 0.f, w0 = 0.f, w1 = 0.f;
      if (gate) {  // gate and up sums of the item's rows (at most 64: two per lane)
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
          const int j = k2 * 32 + lane;
          if (j < rth) {
            const int rlj = j / RH, mj = j % RH;
            float g = 0.f, u = 0.f;
            for (int w = 0; w < WC; ++w) {
              const float* ws = wsum + (s * NCW + rlj * WC + w) * 8;
              g += ws[mj];
              u += ws[RH + mj];
            }
            if (k2 == 0) v0 = g, w0 = u;
            else v1 = g, w1 = u;
          }
        }
      } else {  // the item's RTD row sums (at most 64: two per lane)
        const D1Geo& g = sh_row ? gs : gr;
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
          const int r = k2 * 32 + lane;
          if (r < RTD) {
            const int rl = r % g.NRL, m = r / g.NRL;
            float y = 0.f;
            for (int w = 0; w < g.WC; ++w) y += wsum[(s * NCW + rl * g.WC + w) * 8 + m];
            if (k2 == 0) v0 = y;
            else v1 = y;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // the stage is free; the rest is off the ring's path
      if (gate) {
        const int nc = (sh_row ? a.Fs : a.F) >> 5;
        const int c0 = sh_row ? 0 : has_sh * (a.Fs >> 5) + (e - has_sh) * (a.F >> 5);
        publish_hgroup(a, c0, nc, tile * rth + lane, silu1(v0) * w0, lane < rth, lane);
        if (rth > 32) publish_hgroup(a, c0, nc, tile * rth + 32 + lane, silu1(v1) * w1, 32 + lane < rth, lane);
        __syncwarp();
        if (lane == 0) red_add_release_gpu(&a.ws.hcnt[e], 1u);
      } else {
        float* yp = a.ws.ypart + static_cast<size_t>(e) * H + static_cast<size_t>(tile) * RTD;
        if (lane < RTD) yp[lane] = v0;
        if (32 + lane < RTD) yp[32 + lane] = v1;
        __syncwarp();
        unsigned old = 0;
        if (lane == 0) old = atom_add_acq_rel_gpu(&a.ws.tcnt[tile], 1u);
        old = __shfl_sync(kAll, old, 0);
        // the producer wrote the step's expert count before it issued any
        // down item (every down item comes after the routing)
        if (n_ent < 0) n_ent = *s_nent;
        if (old + 1 == static_cast<unsigned>(n_ent)) {  // every expert's rows of this tile are in
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int r = k2 * 32 + lane;
            if (r < RTD) {
              const size_t row = static_cast<size_t>(tile) * RTD + r;
              float out = 0.f;
              for (int j = 0; j < n_ent; ++j) out += __ldcg(a.ws.ypart + static_cast<size_t>(j) * H + row);
              a.out_bf16[row] = f32_to_bf16_rne(out);
              if (a.out_f32) a.out_f32[row] = out;
            }
          }
          if (lane == 0) a.ws.tcnt[tile] = 0u;
        }
      }
    }
    return;
  }

  // ---------------------------------------------------- consumers
  const int rl = warp / WC, wc = warp % WC, col = wc * 32 + lane;
  const bool gact = warp < NAW && col < C;  // this lane's column of a gate|up item
  float xv[32], sx = 0.f;
#pragma unroll
  for (int m = 0; m < 32; ++m) xv[m] = 0.f;
  if (gact) {
    const uint4* v = reinterpret_cast<const uint4*>(a.x + col * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 t = __ldg(v + i);
      const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) xv[8 * i + 2 * j] = bf16lo(w4[j]), xv[8 * i + 2 * j + 1] = bf16hi(w4[j]);
    }
#pragma unroll
    for (int m = 0; m < 32; ++m) sx += xv[m];
  }
  XChunk X;
  const float scale = make_xchunk_own(xv, X);
  const D1Geo gs = d1_geo(has_sh ? a.Fs : a.F, warp, lane), gr = d1_geo(a.F, warp, lane);

  RingPos pos;
  for (;; pos.next(NST)) {
    const int s = pos.s;
    if (!mbar_wait_sleep_warp(&full[s], pos.ph)) {
      if (lane == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
      break;
    }
    const int code = s_code[s];
    if (code < 0) break;  // the producer ran out of items
    const uint8_t* st = smem + s * SB;
    float* ws = wsum + (s * NCW + warp) * 8;
    if (code & 1) {  // gate|up item
      const uint8_t* stsb = st + 2 * rth * (H / 2);
      float part[R];
#pragma unroll
      for (int m = 0; m < R; ++m) part[m] = 0.f;
      if (gact) {
#pragma unroll
        for (int m = 0; m < R; ++m) {
          const int r = (m < RH) ? (RH * rl + m) : (rth + RH * rl + m - RH);
          const uint4 qv = *reinterpret_cast<const uint4*>(st + r * (H / 2) + col * 16);
          const uint32_t sbw = *reinterpret_cast<const uint32_t*>(stsb + r * (H / 16) + (col >> 1) * 4);
          part[m] = fmaf(bf16lo(sbw) * scale, static_cast<float>(dot_chunk(qv, X)), bf16hi(sbw) * sx);
        }
      }
      constexpr int LPR = 32 / R;  // lanes per row after the butterfly
      float v;
      if constexpr (R == 8) v = bfly8(part, lane);
      else v = bfly4b(part, lane);
      if ((lane & (LPR - 1)) == 0) ws[lane / LPR] = v;
    } else {  // down item: RTD rows of one expert, its h block after the weights
      const bool sh = has_sh && (code >> 20) == 0;
      const D1Geo& g = sh ? gs : gr;
      const int Fe = sh ? a.Fs : a.F, nc = Fe >> 5, rowb = Fe / 2, sbrow = Fe / 16;
      const int RR = RTD / g.NRL;  // rows per thread
      float part[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) part[m] = 0.f;
      if (g.act) {
        const uint8_t* stsb = st + RTD * rowb;
        const uint8_t* xb = stsb + RTD * sbrow;
        const uint4* xw = reinterpret_cast<const uint4*>(xb);
        XChunk Xh;
        const uint4 g0 = xw[0 * nc + g.col], g1 = xw[1 * nc + g.col], g2 = xw[2 * nc + g.col],
                    g3 = xw[3 * nc + g.col];
        Xh.eh[0] = g0.x, Xh.eh[1] = g0.y, Xh.eh[2] = g0.z, Xh.eh[3] = g0.w;
        Xh.el[0] = g1.x, Xh.el[1] = g1.y, Xh.el[2] = g1.z, Xh.el[3] = g1.w;
        Xh.oh[0] = g2.x, Xh.oh[1] = g2.y, Xh.oh[2] = g2.z, Xh.oh[3] = g2.w;
        Xh.ol[0] = g3.x, Xh.ol[1] = g3.y, Xh.ol[2] = g3.z, Xh.ol[3] = g3.w;
        const float p = s_p[s];
        const float4 sc4 = reinterpret_cast<const float4*>(xb + 64 * nc)[g.col];
        const float4 sm4 = reinterpret_cast<const float4*>(xb + 80 * nc)[g.col];
        const float scp[4] = {sc4.x * p, sc4.y * p, sc4.z * p, sc4.w * p};
        const float psx = p * ((sm4.x + sm4.y) + (sm4.z + sm4.w));
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          if (m < RR) {
            const int r = g.rl + g.NRL * m;
            const uint4 qv = *reinterpret_cast<const uint4*>(st + r * rowb + g.col * 16);
            const uint32_t sbw = *reinterpret_cast<const uint32_t*>(stsb + r * sbrow + (g.col >> 1) * 4);
            part[m] = fmaf(bf16lo(sbw), dot_chunk_g(qv, Xh, scp), bf16hi(sbw) * psx);
          }
        }
      }
      const float v = bfly8(part, lane);  // lane L: row (L >> 2) of the warp's column block
      if ((lane & 3) == 0) ws[lane >> 2] = v;
    }
    __syncwarp();  // the lanes' sums before lane 0's arrivals (release at CTA scope)
    if (lane == 0) mbar_arrive(&pdone[s]), mbar_arrive(&empty[s]);
  }
}

size_t ffn_b1_smem_bytes(const LayerArgs& a) { return f1_smem(a.f1_nst, a.f1_stage).total; }

// ============================================================================
// Host side.
// ============================================================================

static int p2floor(int v) {
  int p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}

static int lanes_for(int K, int ncw) {
  const int C = K / 32, WC = (C + 31) / 32;
  return p2floor(std::max(1, ncw / WC));
}

constexpr int kB1SmemBudget = 210 * 1024;

// Row-lanes of the down mapping for an h row of width Fe (as d1_geo).
static int d1_nrl(int Fe) {
  const int C = Fe / 32, WC = (C + 31) / 32;
  return p2floor(std::max(1, kD1Warps / WC));
}

// Geometry of the fused kernel: the largest down item (RTD rows, at most 64,
// a divisor of H and a multiple of 4 and of both widths' row-lanes, at most
// 8 rows per thread) whose stage still leaves a ring of three.  f1_nst = 0
// when none fits (the three-kernel path runs instead).
static void plan_f1(LayerArgs& a, int rth, int smem_optin) {
  a.f1_nst = 0;
  const int H = a.H, Fm = std::max(a.F, a.Fs);
  const int nr = d1_nrl(a.F), ns = a.Fs ? d1_nrl(a.Fs) : nr;
  const int gst = 2 * rth * (H / 2 + H / 16);
  const int budget = std::min(kF1SmemBudget, smem_optin - 1024);
  for (int rt = 64; rt >= 4; --rt) {
    if (H % rt || rt % 4 || rt % nr || rt % ns || rt / nr > 8 || rt / ns > 8) continue;
    if (H / rt > kMaxDim / 8) break;
    const int dst = rt * (Fm / 2 + Fm / 16) + 96 * (Fm / 32);
    const int sb = (std::max(gst, dst) + 127) / 128 * 128;
    // per stage: the stage, its warps' row sums and three barriers
    const int per = sb + (f1_smem(1, 0).total - f1_smem(0, 0).total);
    const int nst = std::min(kF1MaxStages, (budget - f1_smem(0, 0).total) / per);
    if (nst < 3) continue;
    a.f1_rt = rt, a.f1_stage = sb, a.f1_nst = nst;
    return;
  }
}

// Geometry of the B = 1 kernels; false when this layer shape needs the
// general kernels instead (fixed-point h rows too large for shared memory).
bool plan_b1(LayerArgs& a, int num_sms, int smem_optin) {
  const int H = a.H;
  a.gu_nrl = lanes_for(H, kG1Warps);
  // Eight rows per thread when three such stages fit, else four.
  int rows = 8;
  for (;; rows = 4) {
    const int rth = (rows / 2) * a.gu_nrl;
    a.gu_stage = (2 * rth * (H / 2 + H / 16) + 127) / 128 * 128;
    a.gu_nst = std::min(8, (kB1SmemBudget - 4096) / a.gu_stage);
    if (rows == 4 || a.gu_nst >= 3) break;
  }
  a.gu_rows = rows;
  const int rth = (rows / 2) * a.gu_nrl;
  // an item's h values are whole 8-value groups of the fixed-point h, at
  // most two per lane of the warp that writes them
  if (rth % 8 || rth > 64 || a.F % rth || (a.Fs && a.Fs % rth)) return false;
  if (a.gu_nst < 2) return false;

  int nrl_min = lanes_for(a.F, kD1Warps);
  if (a.Fs) nrl_min = std::min(nrl_min, lanes_for(a.Fs, kD1Warps));
  const int rt_cap = kD1Rpt * nrl_min;
  const int Fm = std::max(a.F, a.Fs);
  int best = 4;
  double best_cost = 1e300;
  bool found = false;
  for (int rt = 4; rt <= rt_cap; rt += 4) {
    if (H % rt) continue;
    const int waves = (H / rt + num_sms - 1) / num_sms;
    if (waves > kD1MaxTiles) continue;
    const double cost = static_cast<double>(waves) * rt * (Fm / 2.0 + Fm / 16.0);
    if (cost <= best_cost) best_cost = cost, best = rt, found = true;  // ties: larger tiles
  }
  if (!found) return false;
  a.dn_rt = best;
  a.dn_tiles = H / best;
  a.dn_stage = (best * (Fm / 2 + Fm / 16) + 127) / 128 * 128;
  const int has_sh = a.Fs > 0 ? 1 : 0;
  const int fixed = d1_smem(0, 0, a.k + has_sh, std::max(a.F, a.Fs) / 32).total;
  a.dn_nst = std::min(kD1MaxStages, (kB1SmemBudget - fixed) / a.dn_stage);
  if (a.dn_nst < 2) return false;
  if (gateup_b1_smem_bytes(a, rows) + 1024 > static_cast<size_t>(smem_optin)) return false;
  if (down_b1_smem_bytes(a) + 1024 > static_cast<size_t>(smem_optin)) return false;
  plan_f1(a, rth, smem_optin);
  return true;
}

cudaError_t set_b1_attributes(int smem_optin) {
  const void* fns[] = {(const void*)router_b1_kernel,
                       (const void*)gateup_b1_kernel<4>,
                       (const void*)gateup_b1_kernel<8>, (const void*)down_b1_kernel,
                       (const void*)ffn_b1_kernel<4>, (const void*)ffn_b1_kernel<8>};
  for (const void* f : fns) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, f);
    if (e) return e;
    if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  smem_optin - static_cast<int>(fa.sharedSizeBytes))))
      return e;
  }
  return cudaSuccess;
}

static cudaError_t launch1(const void* fn, int grid, int block, size_t smem, cudaStream_t st, bool pdl,
                           const LayerArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  void* args[] = {const_cast<LayerArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

static cudaError_t mark1(const LayerArgs& a, int i, cudaStream_t st) {
  return a.prof_on ? cudaEventRecord(static_cast<cudaEvent_t>(a.prof[i]), st) : cudaSuccess;
}


static cudaError_t launch_router1(const LayerArgs& a, int num_sms, cudaStream_t st) {
  const int rgrid = std::max(1, std::min((a.E + kR1Rows - 1) / kR1Rows, 2 * num_sms));
  return launch1((const void*)router_b1_kernel, rgrid, kR1Threads, router_b1_smem_bytes(a.E), st,
                 a.x_pdl != 0 && !a.prof_on, a);
}

// Copies n16 16-byte words from src (mapped page-locked host memory) to dst
// (device).  It releases its dependents at once: a single-token router
// launched after it loads its weight rows meanwhile and waits for the copy
// before it reads x.
__global__ void __launch_bounds__(256) stage_x_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int n16) {
  pdl_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += gridDim.x * blockDim.x) dst[i] = src[i];
}

cudaError_t launch_stage_x(const void* src, void* dst, size_t bytes, cudaStream_t st) {
  const int n16 = static_cast<int>(bytes / 16);
  const int grid = std::max(1, std::min(8, (n16 + 255) / 256));
  stage_x_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
  return cudaGetLastError();
}

static cudaError_t launch_gateup1(const LayerArgs& a, int part, int num_sms, cudaStream_t st, bool pdl) {
  LayerArgs b = a;
  b.gu_part = part;
  const void* gu = b.gu_rows == 8 ? (const void*)gateup_b1_kernel<8> : (const void*)gateup_b1_kernel<4>;
  return launch1(gu, num_sms, kG1Threads, gateup_b1_smem_bytes(b, b.gu_rows), st, pdl, b);
}

static cudaError_t launch_down1(const LayerArgs& a, int num_sms, cudaStream_t st, bool pdl) {
  return launch1((const void*)down_b1_kernel, num_sms, (kD1Warps + 1) * 32, down_b1_smem_bytes(a), st, pdl, a);
}

static cudaError_t launch_ffn1(const LayerArgs& a, int num_sms, cudaStream_t st, bool pdl) {
  const void* fn = a.gu_rows == 8 ? (const void*)ffn_b1_kernel<8> : (const void*)ffn_b1_kernel<4>;
  return launch1(fn, num_sms, kF1Threads, ffn_b1_smem_bytes(a), st, pdl, a);
}

// Launches the B = 1 path; `a` already planned by plan_b1.  The router, then
// the fused gate|up + down kernel where it is planned (profile events: the
// router, the fused kernel, nothing), else gate|up and down.
cudaError_t launch_decode_b1(const LayerArgs& a, int num_sms, cudaStream_t st) {
  const bool pdl = !a.prof_on;
  cudaError_t e;
  if (a.f1_nst > 0 && !a.slot_of) {
    if ((e = mark1(a, 0, st)) || (e = launch_router1(a, num_sms, st)) || (e = mark1(a, 1, st)) ||
        (e = launch_ffn1(a, num_sms, st, pdl)) || (e = mark1(a, 2, st)))
      return e;
    return mark1(a, 3, st);
  }
  if ((e = mark1(a, 0, st))) return e;
  if ((e = launch_router1(a, num_sms, st))) return e;
  if ((e = mark1(a, 1, st))) return e;
  if ((e = launch_gateup1(a, 0, num_sms, st, pdl))) return e;
  if ((e = mark1(a, 2, st))) return e;
  if ((e = launch_down1(a, num_sms, st, pdl))) return e;
  return mark1(a, 3, st);
}

// The same step in three parts, for the expert cache: the router; the shared
// expert's gate|up (which runs while the host updates the cache and copies
// the missing records); then the routed experts' gate|up and the down +
// combine kernel.
cudaError_t launch_b1_router(const LayerArgs& a, int num_sms, cudaStream_t st) {
  return launch_router1(a, num_sms, st);
}

cudaError_t launch_b1_shared(const LayerArgs& a, int num_sms, cudaStream_t st) {
  return launch_gateup1(a, 1, num_sms, st, false);
}

cudaError_t launch_b1_routed(const LayerArgs& a, int num_sms, cudaStream_t st) {
  cudaError_t e = launch_gateup1(a, 2, num_sms, st, false);
  return e ? e : launch_down1(a, num_sms, st, true);
}

}  // namespace moe
