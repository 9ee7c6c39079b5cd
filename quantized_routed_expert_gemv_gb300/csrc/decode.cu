// decode.cu -- CUDA-core kernels of the MoE FFN decode step (sm_103a).
//
//   router_kernel   8-bit affine router GEMV -> fp32 logits; the last CTA to
//                   finish runs softmax + warp-shuffle top-k per token and
//                   groups the (token, slot) pairs by expert.
//   gateup_kernel   4-bit gate|up GEMV + SwiGLU for the shared expert and
//                   every active expert; each expert's rows are read once per
//                   step and applied to all of its tokens.  The shared
//                   expert's rows need no routing and are streamed while the
//                   router is still running (programmatic dependent launch).
//   down_kernel     4-bit down GEMV fused with the combine: a CTA owns a row
//                   tile of the output and walks every expert of the step in
//                   a fixed order, accumulating p_i * y_i (and y_shared) in
//                   shared memory, so no partial results leave the SM.
//
// The method follows the TurboFieldfare page, section "Token üretim süreci"
// (router on resident weights, top-8 ids, shared expert computed while
// routed weights are fetched, shared and routed outputs combined; one
// fetched expert serves several rows) and section "Belleği azaltan çalışma
// yapısı" (affine 4-bit group-64 experts, 8-bit router); the record holds
// gate, up and down contiguously as on the WASTE page, section "Disk
// streaming mimarisi".
//
// Weight streaming.  One producer warp per CTA moves each work item's rows
// (codes + scale/bias words, and for `down` the expert's activations) from
// HBM into a ring of shared-memory stages with 1-D bulk copies
// (cp.async.bulk, completion on an mbarrier); the consumer warps compute from
// shared memory and hand the stage back through a second mbarrier.
//
// The GEMV inner loops (float path) are in gemv.cuh.
#include <algorithm>
#include <cfloat>

#include "common.cuh"
#include "gemv.cuh"
#include "kernels.h"

namespace moe {

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Lane 0 waits (bounded) and the result is broadcast to the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(bar, parity) ? 1 : 0;
  return __shfl_sync(kFull, ok, 0) != 0;
}

// ============================================================================
// Router: logits, then (last CTA) top-k, weights and grouping by expert.
// ============================================================================

constexpr int kRouterThreads = 512;
constexpr int kRouterRows = 4;  // rows in flight per iteration
// control words of the multi-token router: per token block, row-block CTAs
// done with its logits; token blocks done with their top-k
constexpr int kCtlTopkDone = 15;
constexpr int kCtlTokenBlock0 = 16;
constexpr int kRouterMaxTokenBlocks = 48;  // ctl[16 .. 63]

// Warp groups: a group of WPR = ceil(H / 512) warps covers a router row (its
// thread c owns 16-byte chunk c, 16 activations); the block's G = 16 / WPR
// groups take different tokens of a pass, so small H keeps every warp busy.
__host__ __device__ inline int router_groups(int H) {
  const int wpr = ((H >> 4) + 31) / 32;
  return (kRouterThreads / 32) / wpr;
}

// Each CTA holds kRouterRows router rows in registers (all loads in flight at
// once) and walks its token passes of NT tokens per group.
template <int NT, int KPL>  // KPL: logit slots per lane of a top-k warp, KPL * 32 >= E
__global__ void __launch_bounds__(kRouterThreads) router_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(16) float rsm[];
  pdl_launch_dependents();
  const int H = a.H, E = a.E, T = a.T, k = a.k;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int NW = kRouterThreads / 32;
  const int nchunk = H >> 4, WPR = (nchunk + 31) / 32, G = NW / WPR;
  const int g = warp / WPR, wi = warp - g * WPR, c = tid - g * WPR * 32;
  const bool act = g < G && c < nchunk;
  float* red = rsm;  // [G][NT][kRouterRows][WPR]

  // The last xq_nconv CTAs convert the tokens; the ones before them compute
  // the logits, so the top-k never waits for a conversion.
  const int nlog = static_cast<int>(gridDim.x) - a.xq_nconv;
  if (static_cast<int>(blockIdx.x) >= nlog) {
    // The few-token fused kernel (decode_bt.cu) reads every token's
    // activations in the fixed-point chunk form of gemv.cuh: these CTAs
    // write them once ([T][4 kinds][C] words, then [T][C] (2^e, plain sum))
    // and count themselves done on ctl[10] (release).
    const int C = H >> 5, n = T * C, ci = static_cast<int>(blockIdx.x) - nlog;
    uint4* xw = reinterpret_cast<uint4*>(a.ws.xq);
    float2* xs = reinterpret_cast<float2*>(a.ws.xq + static_cast<size_t>(T) * C * 64);
    for (int i = ci * kRouterThreads + tid; i < n; i += a.xq_nconv * kRouterThreads) {
      const int t = i / C, c = i - t * C;
      const uint4* v = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * H + c * 32);
      float xv[32], sx = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 w4 = __ldg(v + j);
        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int b = 0; b < 4; ++b) xv[8 * j + 2 * b] = bf16lo(w[b]), xv[8 * j + 2 * b + 1] = bf16hi(w[b]);
      }
#pragma unroll
      for (int m = 0; m < 32; ++m) sx += xv[m];
      XChunk X;
      const float scale = make_xchunk_own(xv, X);
      xw[(static_cast<size_t>(t) * 4 + 0) * C + c] = make_uint4(X.eh[0], X.eh[1], X.eh[2], X.eh[3]);
      xw[(static_cast<size_t>(t) * 4 + 1) * C + c] = make_uint4(X.el[0], X.el[1], X.el[2], X.el[3]);
      xw[(static_cast<size_t>(t) * 4 + 2) * C + c] = make_uint4(X.oh[0], X.oh[1], X.oh[2], X.oh[3]);
      xw[(static_cast<size_t>(t) * 4 + 3) * C + c] = make_uint4(X.ol[0], X.ol[1], X.ol[2], X.ol[3]);
      xs[static_cast<size_t>(t) * C + c] = make_float2(scale, sx);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) red_add_release_gpu(&a.ws.ctl[10], 1u);
    return;
  }

  // The logits grid is (row blocks of kRouterRows experts) x (token blocks):
  // a CTA loads its router rows once and walks its share of the token passes.
  const int RB = (E + kRouterRows - 1) / kRouterRows;
  const int TB = max(1, nlog / RB);
  const int rb = blockIdx.x % RB, tb = blockIdx.x / RB;
  const int er0 = rb * kRouterRows;
  const int TP = NT * G;  // tokens per pass
  const int npass = (T + TP - 1) / TP, ppb = (npass + TB - 1) / TB;
  const int p_lo = tb * ppb, p_hi = min(npass, p_lo + ppb);
  uint4 q[kRouterRows];
  uint32_t sbw[kRouterRows];
#pragma unroll
  for (int r = 0; r < kRouterRows; ++r) {
    q[r] = make_uint4(0, 0, 0, 0), sbw[r] = 0;
    if (act && er0 + r < E && tb < TB) {
      q[r] = __ldg(reinterpret_cast<const uint4*>(a.rcodes + static_cast<size_t>(er0 + r) * H) + c);
      sbw[r] = __ldg(a.rsb + static_cast<size_t>(er0 + r) * (H >> 6) + (c >> 2));
    }
  }
  const int nout = G * NT * kRouterRows;  // logits per pass, one per thread tid < nout
  float beta_r = 0.f;
  if (tid < nout && a.beta && er0 + tid % kRouterRows < E) beta_r = __ldg(a.beta + er0 + tid % kRouterRows);

  // The activations of the next token pass are loaded while this one is
  // computed: raw bf16 words, two uint4 per token.
  uint4 xr[NT][2];
  auto load_x = [&](int pi) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      xr[t][0] = xr[t][1] = make_uint4(0, 0, 0, 0);
      const int tok = pi * TP + g * NT + t;
      if (act && pi < p_hi && tok < T) {
        const uint4* xp = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(tok) * H + c * 16);
        xr[t][0] = __ldg(xp), xr[t][1] = __ldg(xp + 1);
      }
    }
  };
  load_x(p_lo);
  for (int pi = p_lo; pi < p_hi; ++pi) {
    const int t0 = pi * TP + g * NT;  // this group's first token of the pass
    float2 X[NT][8];
    float SX[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      SX[t] = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) X[t][j] = make_float2(0.f, 0.f);
      if (act && t0 + t < T) {
        const uint32_t xw[8] = {xr[t][0].x, xr[t][0].y, xr[t][0].z, xr[t][0].w,
                                xr[t][1].x, xr[t][1].y, xr[t][1].z, xr[t][1].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float lo = bf16lo(xw[j]), hi = bf16hi(xw[j]);
          X[t][j] = make_float2(lo * byte_scale((2 * j) & 3), hi * byte_scale((2 * j + 1) & 3));
          SX[t] += lo;
          SX[t] += hi;
        }
      }
    }
    load_x(pi + 1);  // in flight while this pass is computed
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int r = 0; r < kRouterRows; ++r) {
        const float p = fmaf(bf16lo(sbw[r]) * 0x1p64f, dot16_u8(q[r], X[t]), bf16hi(sbw[r]) * SX[t]);
        const float v = warp_sum(p);
        if (lane == 0 && g < G) red[((g * NT + t) * kRouterRows + r) * WPR + wi] = v;
      }
    }
    __syncthreads();
    if (tid < nout) {  // tid = (group, token, row)
      const int gg = tid / (NT * kRouterRows), t = (tid / kRouterRows) % NT, r = tid % kRouterRows;
      const int tok = pi * TP + gg * NT + t;
      if (tok < T && er0 + r < E) {
        float v = 0.f;
        for (int w = 0; w < WPR; ++w) v += red[tid * WPR + w];
        a.ws.logits[static_cast<size_t>(tok) * E + er0 + r] = v + beta_r;
      }
    }
    __syncthreads();
  }

  // ---- top-k per token block, then grouping by the last token block ------
  // The last of the RB row-block CTAs of token block tb to finish its
  // logits takes the top-k of the block's tokens (every logit of them is
  // written by then); the last token block to finish its top-k groups every
  // token's pairs by expert.  Both counters go back to zero in the CTA that
  // completes them.
  __shared__ int s_last;
  unsigned* const tb_done = &a.ws.ctl[kCtlTokenBlock0 + tb];
  unsigned* const tk_done = &a.ws.ctl[kCtlTopkDone];
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(tb_done, 1u) == static_cast<unsigned>(RB - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) *tb_done = 0u;

  unsigned* sel = reinterpret_cast<unsigned*>(rsm + NW * E);      // [E][4] token bitmasks
  int* s_off = reinterpret_cast<int*>(sel + 4 * E);               // [E] pair offsets
  int* s_ids = s_off + E;                                         // [T*k]
  int* s_scan = s_ids + kMaxTokens * kMaxTopK;                    // [2*NW] scan scratch
  const int t_lo = min(T, p_lo * TP), t_hi = min(T, p_hi * TP);  // this token block's tokens

  // One warp per token.  Lane l holds the keys of experts l, l+32, ... in
  // registers (a logit's IEEE bits mapped to an order-preserving unsigned;
  // 0 marks a taken or absent expert) and its best key; a round takes the
  // warp's maximum (ties: the lower id) and only the winner's lane rescans.
  // The warp's next token's logits are loaded while this one is selected.
  float lnext[KPL];
  auto load_logits = [&](int t) {
#pragma unroll
    for (int s2 = 0; s2 < KPL; ++s2) {
      const int e = s2 * 32 + lane;
      lnext[s2] = (t < t_hi && e < E) ? __ldcg(a.ws.logits + static_cast<size_t>(t) * E + e) : 0.f;
    }
  };
  load_logits(t_lo + warp);
  for (int t = t_lo + warp; t < t_hi; t += NW) {
    uint32_t key[KPL];
#pragma unroll
    for (int s2 = 0; s2 < KPL; ++s2) {
      const int e = s2 * 32 + lane;
      uint32_t kk = 0u;
      if (e < E) {
        const uint32_t u = __float_as_uint(lnext[s2]);
        kk = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
      }
      key[s2] = kk;
    }
    load_logits(t + NW);
    uint32_t bk = 0u;
    int bs = 0;
#pragma unroll
    for (int s2 = 0; s2 < KPL; ++s2)
      if (key[s2] > bk) bk = key[s2], bs = s2;
    float myl = 0.f;
    int myi = 0;
    for (int i = 0; i < k; ++i) {
      const uint32_t top = __reduce_max_sync(kFull, bk);
      const unsigned win = __reduce_min_sync(
          kFull, (bk == top && top != 0u) ? static_cast<unsigned>(bs * 32 + lane) : 0xFFFFFFFFu);
      int bi = static_cast<int>(win);
      if (bi >= E) {  // only reachable with non-finite logits (outside the contract)
        if (lane == 0) latch_error(&a.ws.ctl[0], kErrRange);
        bi = i;
      }
      if (lane == i) myi = bi, myl = __uint_as_float((top & 0x80000000u) ? (top & 0x7FFFFFFFu) : ~top);
      if ((bi & 31) == lane) {
        const int ws = bi >> 5;
        bk = 0u, bs = 0;
#pragma unroll
        for (int s2 = 0; s2 < KPL; ++s2) {
          if (s2 == ws) key[s2] = 0u;
          if (key[s2] > bk) bk = key[s2], bs = s2;
        }
      }
    }
    const float lmax = __shfl_sync(kFull, myl, 0);
    const float ex = (lane < k) ? expf(myl - lmax) : 0.f;
    const float z = warp_sum(ex);
    if (lane < k) {
      a.ids[t * k + lane] = myi;
      a.weights[t * k + lane] = ex / z;
      if (a.ids_host) a.ids_host[t * k + lane] = myi, a.weights_host[t * k + lane] = ex / z;
    }
    __syncwarp();
  }

  // the last token block: every token's ids are in; group the pairs (with
  // one token block this CTA took every token's top-k itself)
  if (TB > 1) {
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(tk_done, 1u) == static_cast<unsigned>(TB - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid == 0) *tk_done = 0u;
  } else {
    __syncthreads();
  }

  for (int i = tid; i < 4 * E; i += kRouterThreads) sel[i] = 0u;
  __syncthreads();
  for (int p = tid; p < T * k; p += kRouterThreads) {
    int e = __ldcg(a.ids + p);
    if (e < 0 || e >= E) e = 0;  // (a range error was latched where it arose)
    const int t = p / k;
    s_ids[p] = e;
    atomicOr(&sel[e * 4 + (t >> 5)], 1u << (t & 31));
  }
  __syncthreads();

  // counts and exclusive scans over experts (pairs, active experts)
  const int ept = (E + kRouterThreads - 1) / kRouterThreads;
  const int e0 = tid * ept, e1 = min(e0 + ept, E);
  int c_loc = 0, a_loc = 0;
  for (int e = e0; e < e1; ++e) {
    const int c = __popc(sel[4 * e]) + __popc(sel[4 * e + 1]) + __popc(sel[4 * e + 2]) +
                  __popc(sel[4 * e + 3]);
    c_loc += c;
    a_loc += (c > 0);
  }
  int c_inc = c_loc, a_inc = a_loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int cu = __shfl_up_sync(kFull, c_inc, o);
    const int au = __shfl_up_sync(kFull, a_inc, o);
    if (lane >= o) c_inc += cu, a_inc += au;
  }
  if (lane == 31) s_scan[warp] = c_inc, s_scan[NW + warp] = a_inc;
  __syncthreads();
  int c_base = 0, a_base = 0;
  for (int w = 0; w < warp; ++w) c_base += s_scan[w], a_base += s_scan[NW + w];
  int c_run = c_base + c_inc - c_loc, a_run = a_base + a_inc - a_loc;
  for (int e = e0; e < e1; ++e) {
    const int c = __popc(sel[4 * e]) + __popc(sel[4 * e + 1]) + __popc(sel[4 * e + 2]) +
                  __popc(sel[4 * e + 3]);
    s_off[e] = c_run;
    if (c > 0) {
      a.ws.act_expert[a_run] = e;
      a.ws.act_off[a_run] = c_run;
      a.ws.act_cnt[a_run] = c;
      ++a_run;
    }
    c_run += c;
  }
  if (tid == kRouterThreads - 1) *a.ws.n_act = a_run;
  __syncthreads();

  for (int p = tid; p < T * k; p += kRouterThreads) {
    const int t = p / k, e = s_ids[p];
    int rank = 0;
    for (int w = 0; w < (t >> 5); ++w) rank += __popc(sel[4 * e + w]);
    rank += __popc(sel[4 * e + (t >> 5)] & ((1u << (t & 31)) - 1u));
    const int pos = s_off[e] + rank;
    a.ws.pair_token[pos] = t;
    a.ws.pair_slot[pos] = p;
  }
}

// ============================================================================
// Shared machinery of the two expert GEMV kernels.
// ============================================================================

struct Entry {     // one expert's work this step
  const uint8_t* rec;
  const RecordOffsets* off;  // points into the __grid_constant__ kernel parameter
  int Fe;          // FFN width of this expert (F or Fs)
  int ntok;        // tokens routed to it
  int pair0;       // first (expert, token) pair -- its h row
  int shared;      // 1 for the shared expert
  int expert;      // routed expert id (-1 for the shared expert)
  int slot;        // slot (or expert index) its record is read from
};

__device__ __forceinline__ Entry get_entry(const LayerArgs& a, int idx, int has_sh) {
  Entry en;
  if (has_sh && idx == 0) {
    en.rec = a.shared, en.off = &a.off_s, en.Fe = a.Fs, en.ntok = a.T, en.pair0 = 0;
    en.shared = 1, en.expert = -1, en.slot = -1;
    return en;
  }
  const int i = idx - has_sh;
  int e = a.ws.act_expert[i];
  int cnt = a.ws.act_cnt[i];
  if (e < 0 || e >= a.E) e = 0;
  if (cnt < 0 || cnt > a.T) cnt = 0;
  int slot = e;
  if (a.slot_of) {  // residency: a slot outside the pool is never read
    slot = a.slot_of[e];
    if (slot < 0 || slot >= a.n_slots) latch_error(&a.ws.ctl[0], kErrResidency), slot = 0;
  }
  en.rec = a.records + static_cast<size_t>(slot) * a.off_r.stride;
  en.off = &a.off_r, en.Fe = a.F, en.ntok = cnt, en.pair0 = a.ws.act_off[i];
  en.shared = 0, en.expert = e;
  en.slot = slot;
  return en;
}

__device__ __forceinline__ int read_n_act(const LayerArgs& a) {
  const int n = *reinterpret_cast<volatile int*>(a.ws.n_act);
  return n < 0 ? 0 : (n > a.E ? a.E : n);
}

// ============================================================================
// gate|up + SwiGLU.  Consumer warp w covers 32 consecutive 16-byte columns
// (wc = w % WC) of row-lane rl = w / WC; every thread owns one column and
// gate rows {2rl, 2rl+1} plus up rows {2rl, 2rl+1} of the item, so the
// SwiGLU pairs meet after one cross-warp sum.  Item = rth = 2*NRL gate rows
// and the same up rows of one expert; the shared expert's items come first.
// ============================================================================

template <int NTOK, int NCW>
__global__ void __launch_bounds__((NCW + 1) * 32, 1) gateup_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NCT = NCW * 32;
  const int H = a.H, C = H >> 5, WC = (C + 31) >> 5, NRL = a.gu_nrl, rth = 2 * NRL;
  const int NST = a.gu_nst, SB = a.gu_stage;
  float* wsum = reinterpret_cast<float*>(smem + NST * SB);  // [2][NTOK][NCW][4]
  uint64_t* full = reinterpret_cast<uint64_t*>(wsum + 2 * NTOK * NCW * 4);
  uint64_t* empty = full + NST;
  volatile int* s_abort = reinterpret_cast<volatile int*>(empty + NST);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&full[s], 1), mbar_init(&empty[s], NCW);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_launch_dependents();

  const int has_sh = a.Fs > 0 ? 1 : 0;
  const int tiles_s = has_sh ? a.Fs / rth : 0, tiles_r = a.F / rth;
  // Item i < tiles_s: shared expert tile i (no routing needed).  Later items
  // need the router's output; n_items is only known after pdl_wait().

  if (warp == NCW) {  // ---------------- producer warp
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0, n_items = tiles_s;
      bool waited = false;
      for (int i = blockIdx.x;; i += gridDim.x, ++it) {
        if (i >= tiles_s && !waited) {
          pdl_wait();
          waited = true;
          n_items = tiles_s + read_n_act(a) * tiles_r;
        }
        if (i >= n_items) break;
        const int s = it % NST;
        if (it >= NST && !mbar_wait(&empty[s], ((it / NST) - 1) & 1)) {
          latch_error(&a.ws.ctl[0], kErrTimeout);
          break;
        }
        const int idx = i < tiles_s ? 0 : has_sh + (i - tiles_s) / tiles_r;
        const int tile = i < tiles_s ? i : (i - tiles_s) % tiles_r;
        const Entry en = get_entry(a, idx, has_sh);
        if (!en.shared && a.slot_tag && a.slot_tag[en.slot] != en.expert)
          latch_error(&a.ws.ctl[0], kErrResidency);
        const size_t j0 = static_cast<size_t>(tile) * rth;
        const uint32_t cb = rth * (H / 2), sbb = rth * (H / 16);
        uint8_t* st = smem + s * SB;
        mbar_arrive_expect_tx(&full[s], 2 * cb + 2 * sbb);
        bulk_g2s(st, en.rec + en.off->gate_codes + j0 * (H / 2), cb, &full[s], pol);
        bulk_g2s(st + cb, en.rec + en.off->up_codes + j0 * (H / 2), cb, &full[s], pol);
        bulk_g2s(st + 2 * cb, en.rec + en.off->gate_sb + j0 * (H / 16), sbb, &full[s], pol);
        bulk_g2s(st + 2 * cb + sbb, en.rec + en.off->up_sb + j0 * (H / 16), sbb, &full[s], pol);
      }
      for (int j = max(0, it - NST); j < it; ++j)  // every issued copy lands before exit
        if (!mbar_wait(&full[j % NST], (j / NST) & 1)) latch_error(&a.ws.ctl[0], kErrTimeout);
    }
    return;
  }

  // ---------------------------------------------------- consumer warps
  const int rl = warp / WC, wc = warp % WC, col = wc * 32 + lane;
  const bool active = (rl < NRL) && (col < C);
  float2 X[NTOK][16];
  float SX[NTOK];
  const bool single = (a.T == 1);  // every entry's only token is token 0
  if (single) {
    if (active) load_x_bf16(a.x + col * 32, X[0], SX[0]);
    else zero_x(X[0], SX[0]);
  }

  int it = 0, n_items = tiles_s;
  bool waited = false, abort_all = false;
  for (int i = blockIdx.x;; i += gridDim.x, ++it) {
    if (i >= tiles_s && !waited) {
      pdl_wait();
      waited = true;
      n_items = tiles_s + read_n_act(a) * tiles_r;
    }
    if (i >= n_items) break;
    const int s = it % NST;
    if (!warp_wait(&full[s], (it / NST) & 1, lane)) *s_abort = 1;
    const int idx = i < tiles_s ? 0 : has_sh + (i - tiles_s) / tiles_r;
    const int tile = i < tiles_s ? i : (i - tiles_s) % tiles_r;
    const Entry en = get_entry(a, idx, has_sh);
    const uint8_t* st = smem + s * SB;
    const uint8_t* stsb = st + 2 * rth * (H / 2);
    float* hout = en.shared ? a.ws.h_shared : a.ws.h;
    const int j0 = tile * rth;
    const int rows[4] = {2 * rl, 2 * rl + 1, rth + 2 * rl, rth + 2 * rl + 1};

    for (int tg = 0; tg < en.ntok; tg += NTOK) {
      const int buf = (it + tg / NTOK) & 1;
      if (!single) {
#pragma unroll
        for (int t = 0; t < NTOK; ++t) {
          if (active && tg + t < en.ntok) {
            const int tok = en.shared ? tg + t : a.ws.pair_token[en.pair0 + tg + t];
            load_x_bf16(a.x + static_cast<size_t>(tok) * H + col * 32, X[t], SX[t]);
          } else {
            zero_x(X[t], SX[t]);
          }
        }
      }
      float part[NTOK][4];
      if (active) {
        uint4 q[4];
        uint32_t sbw[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          q[r] = *reinterpret_cast<const uint4*>(st + rows[r] * (H / 2) + col * 16);
          sbw[r] = *reinterpret_cast<const uint32_t*>(stsb + rows[r] * (H / 16) + (col >> 1) * 4);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float sc = bf16lo(sbw[r]) * 0x1p64f, bi = bf16hi(sbw[r]);
#pragma unroll
          for (int t = 0; t < NTOK; ++t) part[t][r] = fmaf(sc, dot32(q[r], X[t]), bi * SX[t]);
        }
      } else {
#pragma unroll
        for (int t = 0; t < NTOK; ++t)
#pragma unroll
          for (int r = 0; r < 4; ++r) part[t][r] = 0.f;
      }
      if (tg + NTOK >= en.ntok) {  // last pass over this stage: hand it back
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
#pragma unroll
      for (int t = 0; t < NTOK; ++t) {
        const float v = bfly4(part[t][0], part[t][1], part[t][2], part[t][3], lane);
        if ((lane & 7) == 0) wsum[((buf * NTOK + t) * NCW + warp) * 4 + (lane >> 3)] = v;
      }
      if (named_bar_or(1, NCT, *s_abort != 0)) {
        abort_all = true;
        break;
      }
      // SwiGLU on the highest-numbered threads: warps past NRL*WC have no
      // column of their own, so the epilogue costs the busy warps nothing.
      for (int q = NCT - 1 - tid; q < NTOK * rth; q += NCT) {
        const int t = q / rth, j = q % rth;
        if (tg + t < en.ntok) {
          const int rlj = j >> 1, jj = j & 1;
          float g = 0.f, u = 0.f;
          for (int w = 0; w < WC; ++w) {
            const float* ws = wsum + ((buf * NTOK + t) * NCW + rlj * WC + w) * 4;
            g += ws[jj];
            u += ws[2 + jj];
          }
          const int hrow = en.shared ? (tg + t) : (en.pair0 + tg + t);
          hout[static_cast<size_t>(hrow) * en.Fe + h_index(j0 + j, en.Fe)] = silu_f(g) * u;
        }
      }
    }
    if (abort_all) {
      if (tid == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
      break;
    }
    if (en.ntok == 0) {  // cannot happen for a listed expert; keep the ring consistent
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  if (!waited) pdl_wait();
}

// ============================================================================
// down + combine.  A CTA owns row tiles of the output (rt rows of H) and, for
// each tile, walks the shared expert then every active expert in ascending
// id order; one item = the tile's rows of one expert for up to NTOK of its
// tokens, staged together with those tokens' h rows.  The weighted sum
// out = y_shared + sum_i p_i y_i builds up in shared memory in that fixed
// order and is written once per tile.
// ============================================================================

template <int NTOK, int NCW>
__global__ void __launch_bounds__((NCW + 1) * 32, 1) down_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NCT = NCW * 32;
  const int H = a.H, RT = a.dn_rt, NST = a.dn_nst, SB = a.dn_stage, T = a.T, k = a.k;
  float* wsum = reinterpret_cast<float*>(smem + NST * SB);  // [2][NTOK][NCW][4]
  float* acc = wsum + 2 * NTOK * NCW * 4;                   // [T][RT]
  uint64_t* full = reinterpret_cast<uint64_t*>(acc + T * RT + ((T * RT) & 1));
  uint64_t* empty = full + NST;
  volatile int* s_abort = reinterpret_cast<volatile int*>(empty + NST);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&full[s], 1), mbar_init(&empty[s], NCW);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int q = tid; q < T * RT; q += blockDim.x) acc[q] = 0.f;
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();  // h of every expert is ready past this point

  const int has_sh = a.Fs > 0 ? 1 : 0;
  const int n_ent = read_n_act(a) + has_sh;
  const int n_tiles = a.dn_tiles;

  if (warp == NCW) {  // ---------------- producer warp
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      bool stop = false;
      for (int tile = blockIdx.x; tile < n_tiles && !stop; tile += gridDim.x) {
        const size_t r0 = static_cast<size_t>(tile) * RT;
        for (int idx = 0; idx < n_ent && !stop; ++idx) {
          const Entry en = get_entry(a, idx, has_sh);
          if (!en.shared && a.slot_tag && a.slot_tag[en.slot] != en.expert)
            latch_error(&a.ws.ctl[0], kErrResidency);
          const float* hb = en.shared ? a.ws.h_shared : a.ws.h + static_cast<size_t>(en.pair0) * en.Fe;
          for (int tg = 0; tg < en.ntok; tg += NTOK, ++it) {
            const int s = it % NST;
            if (it >= NST && !mbar_wait(&empty[s], ((it / NST) - 1) & 1)) {
              latch_error(&a.ws.ctl[0], kErrTimeout);
              stop = true;
              break;
            }
            const int ntg = min(NTOK, en.ntok - tg);
            const uint32_t cb = RT * (en.Fe / 2), sbb = RT * (en.Fe / 16), hbytes = ntg * en.Fe * 4;
            uint8_t* st = smem + s * SB;
            mbar_arrive_expect_tx(&full[s], cb + sbb + hbytes);
            bulk_g2s(st, en.rec + en.off->down_codes + r0 * (en.Fe / 2), cb, &full[s], pol);
            bulk_g2s(st + cb, en.rec + en.off->down_sb + r0 * (en.Fe / 16), sbb, &full[s], pol);
            bulk_g2s(st + cb + sbb, hb + static_cast<size_t>(tg) * en.Fe, hbytes, &full[s]);
          }
        }
      }
      for (int j = max(0, it - NST); j < it; ++j)
        if (!mbar_wait(&full[j % NST], (j / NST) & 1)) latch_error(&a.ws.ctl[0], kErrTimeout);
    }
    return;
  }

  // ---------------------------------------------------- consumer warps
  int it = 0;
  bool abort = false;
  for (int tile = blockIdx.x; tile < n_tiles && !abort; tile += gridDim.x) {
    const int r0 = tile * RT;
    for (int idx = 0; idx < n_ent && !abort; ++idx) {
      const Entry en = get_entry(a, idx, has_sh);
      const int C = en.Fe >> 5, WC = (C + 31) >> 5;
      int NRL = NCW / WC;
      while (NRL & (NRL - 1)) NRL &= NRL - 1;  // power of two
      const int rl = warp / WC, wc = warp % WC, col = wc * 32 + lane;
      const bool active = (rl < NRL) && (col < C);
      for (int tg = 0; tg < en.ntok; tg += NTOK, ++it) {
        const int s = it % NST, buf = it & 1;
        if (!warp_wait(&full[s], (it / NST) & 1, lane)) *s_abort = 1;
        const int ntg = min(NTOK, en.ntok - tg);
        const uint8_t* st = smem + s * SB;
        const uint8_t* stsb = st + RT * (en.Fe / 2);
        const float* sth = reinterpret_cast<const float*>(stsb + RT * (en.Fe / 16));
        float part[NTOK][4];
#pragma unroll
        for (int t = 0; t < NTOK; ++t)
#pragma unroll
          for (int m = 0; m < 4; ++m) part[t][m] = 0.f;
        if (active) {
          float2 X[NTOK][16];
          float SX[NTOK];
#pragma unroll
          for (int t = 0; t < NTOK; ++t) {
            if (t < ntg) load_h_smem(sth + t * en.Fe, C, col, X[t], SX[t]);
            else zero_x(X[t], SX[t]);
          }
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int r = rl + NRL * m;
            if (r < RT) {
              const uint4 q = *reinterpret_cast<const uint4*>(st + r * (en.Fe / 2) + col * 16);
              const uint32_t sbw = *reinterpret_cast<const uint32_t*>(stsb + r * (en.Fe / 16) + (col >> 1) * 4);
              const float sc = bf16lo(sbw) * 0x1p64f, bi = bf16hi(sbw);
#pragma unroll
              for (int t = 0; t < NTOK; ++t) part[t][m] = fmaf(sc, dot32(q, X[t]), bi * SX[t]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
        for (int t = 0; t < NTOK; ++t) {
          const float v = bfly4(part[t][0], part[t][1], part[t][2], part[t][3], lane);
          if ((lane & 7) == 0) wsum[((buf * NTOK + t) * NCW + warp) * 4 + (lane >> 3)] = v;
        }
        if (named_bar_or(1, NCT, *s_abort != 0)) {
          abort = true;
          break;
        }
        // bfly4 leaves the thread's row m (row rl + NRL*m of the tile) at slot m.
        for (int q = tid; q < ntg * RT; q += NCT) {
          const int t = q / RT, r = q % RT;
          const int rlr = r % NRL, m = r / NRL;
          float y = 0.f;
          for (int w = 0; w < WC; ++w) y += wsum[((buf * NTOK + t) * NCW + rlr * WC + w) * 4 + m];
          int tok;
          float p;
          if (en.shared) {
            tok = tg + t, p = 1.f;
          } else {
            const int slot = a.ws.pair_slot[en.pair0 + tg + t];
            tok = slot / k, p = a.weights[slot];
          }
          acc[tok * RT + r] = fmaf(p, y, acc[tok * RT + r]);
        }
      }
    }
    if (named_bar_or(1, NCT, abort)) break;  // every expert of this tile has been added
    for (int q = tid; q < T * RT; q += NCT) {
      const int t = q / RT, r = q % RT;
      const float v = acc[q];
      a.out_bf16[static_cast<size_t>(t) * H + r0 + r] = f32_to_bf16_rne(v);
      if (a.out_f32) a.out_f32[static_cast<size_t>(t) * H + r0 + r] = v;
      acc[q] = 0.f;
    }
  }
  if (abort && tid == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
}

// ============================================================================
// Host side: geometry, shared-memory sizes, launches.
// ============================================================================

static int pow2_floor(int v) {
  int p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}

// Row-lanes of a GEMV whose input width is K, for `ncw` consumer warps.
static int row_lanes(int K, int ncw) {
  const int C = K / 32, WC = (C + 31) / 32;
  return pow2_floor(std::max(1, ncw / WC));
}

static constexpr int kSmemBudget = 200 * 1024;  // pipeline stages per CTA

// Per-launch geometry: gate|up rows per item and stage count; the down row
// tile (a multiple of 4 dividing H, at most 4 rows per thread for every
// expert width, two or more waves of tiles when H allows) and stage count.
void plan_decode(LayerArgs& a, int num_sms, int ncw_gateup, int ncw_down, int ntok) {
  const int H = a.H;
  a.gu_nrl = row_lanes(H, ncw_gateup);
  const int rth = 2 * a.gu_nrl;
  a.gu_stage = (2 * rth * (H / 2 + H / 16) + 127) / 128 * 128;
  a.gu_nst = std::max(2, std::min(8, kSmemBudget / a.gu_stage));

  int nrl_min = row_lanes(a.F, ncw_down);
  if (a.Fs) nrl_min = std::min(nrl_min, row_lanes(a.Fs, ncw_down));
  const int rt_cap = 4 * nrl_min;
  const int Fm = std::max(a.F, a.Fs);
  // Busiest CTA's bytes: waves of tiles x (rt weight rows + the staged h row).
  int best = 4;
  double best_cost = 1e300;
  for (int rt = 4; rt <= rt_cap; rt += 4) {
    if (H % rt) continue;
    const double waves = static_cast<double>((H / rt + num_sms - 1) / num_sms);
    const double cost = waves * (rt * (Fm / 2.0 + Fm / 16.0) + ntok * Fm * 4.0);
    if (cost < best_cost) best_cost = cost, best = rt;
  }
  a.dn_rt = best;
  a.dn_tiles = H / best;
  a.dn_stage = (best * (Fm / 2 + Fm / 16) + ntok * Fm * 4 + 127) / 128 * 128;
  a.dn_nst = std::max(2, std::min(8, kSmemBudget / a.dn_stage));
}

size_t router_smem_bytes(int E) {
  constexpr int NW = kRouterThreads / 32;
  const size_t red = static_cast<size_t>(4) * kRouterRows * NW * 4;
  const size_t topk = static_cast<size_t>(NW * E) * 4 + static_cast<size_t>(4 * E) * 4 +
                      static_cast<size_t>(E) * 4 + static_cast<size_t>(kMaxTokens * kMaxTopK) * 4 +
                      2 * NW * 4;
  return std::max(red, topk);
}

size_t gateup_smem_bytes(const LayerArgs& a, int ntok, int ncw) {
  return static_cast<size_t>(a.gu_nst) * a.gu_stage + static_cast<size_t>(2 * ntok * ncw * 4) * 4 +
         2 * a.gu_nst * 8 + 16;
}

size_t down_smem_bytes(const LayerArgs& a, int ntok, int ncw) {
  return static_cast<size_t>(a.dn_nst) * a.dn_stage + static_cast<size_t>(2 * ntok * ncw * 4) * 4 +
         static_cast<size_t>(a.T * a.dn_rt + 2) * 4 + 2 * a.dn_nst * 8 + 16;
}

static cudaError_t launch_ex(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             bool pdl, const LayerArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
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

// Opt every kernel in to the device's full dynamic shared memory once, so
// layers of different shapes opened in any order all launch.
cudaError_t set_decode_attributes(int smem_optin) {
  const void* fns[] = {(const void*)router_kernel<1, 4>,  (const void*)router_kernel<1, 8>,
                       (const void*)router_kernel<1, 16>, (const void*)router_kernel<1, 32>,
                       (const void*)router_kernel<2, 4>,  (const void*)router_kernel<2, 8>,
                       (const void*)router_kernel<2, 16>, (const void*)router_kernel<2, 32>,
                       (const void*)gateup_kernel<1, 16>, (const void*)gateup_kernel<4, 7>,
                       (const void*)down_kernel<1, 8>,    (const void*)down_kernel<4, 7>};
  for (const void* f : fns) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, f);
    if (e) return e;
    const int dyn = smem_optin - static_cast<int>(fa.sharedSizeBytes);
    if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn))) return e;
  }
  return cudaSuccess;
}

// Largest dynamic shared memory any decode launch of this layer can need.
size_t decode_smem_need(const LayerArgs& base, int num_sms) {
  LayerArgs a = base;
  a.T = kMaxTokens;
  size_t need = router_smem_bytes(a.E);
  plan_decode(a, num_sms, 16, 8, 1);
  need = std::max({need, gateup_smem_bytes(a, 1, 16), down_smem_bytes(a, 1, 8)});
  plan_decode(a, num_sms, 7, 7, 4);
  need = std::max({need, gateup_smem_bytes(a, 4, 7), down_smem_bytes(a, 4, 7)});
  return need;
}

static cudaError_t mark(const LayerArgs& a, int i, cudaStream_t st) {
  return a.prof_on ? cudaEventRecord(static_cast<cudaEvent_t>(a.prof[i]), st) : cudaSuccess;
}

// Router grid: row blocks x token blocks.
// CTAs of the router: row blocks x token blocks, up to two waves (the kernel
// takes 128 registers a thread, one CTA per SM): more token blocks shorten
// each CTA's serial token passes.
// Decode batches of up to 16 tokens take one token block: one wave of CTAs
// (a second wave started up to 9 us late at E = 512) and one CTA for every
// token's top-k and the grouping, with no second completion count.
int decode_router_grid(const LayerArgs& a, int num_sms) {
  const int nt = a.T == 1 ? 1 : 2;
  const int rb = (a.E + kRouterRows - 1) / kRouterRows;
  const int tp = nt * router_groups(a.H);  // tokens per pass of a CTA
  if (a.T <= 16) return rb;
  const int tb = std::max(1, std::min({(a.T + tp - 1) / tp, (2 * num_sms) / rb, kRouterMaxTokenBlocks}));
  return rb * tb;
}

static cudaError_t launch_router_g(const LayerArgs& a, int num_sms, cudaStream_t st) {
  const bool one = (a.T == 1);
  const int rgrid = decode_router_grid(a, num_sms);
  const int kpl = a.E <= 128 ? 4 : a.E <= 256 ? 8 : a.E <= 512 ? 16 : 32;
  const void* fn;
  if (one)
    fn = kpl == 4 ? (const void*)router_kernel<1, 4> : kpl == 8 ? (const void*)router_kernel<1, 8>
       : kpl == 16 ? (const void*)router_kernel<1, 16> : (const void*)router_kernel<1, 32>;
  else
    fn = kpl == 4 ? (const void*)router_kernel<2, 4> : kpl == 8 ? (const void*)router_kernel<2, 8>
       : kpl == 16 ? (const void*)router_kernel<2, 16> : (const void*)router_kernel<2, 32>;
  // the conversion CTAs (few-token fused path) follow the logits CTAs
  return launch_ex(fn, dim3(rgrid + a.xq_nconv), dim3(kRouterThreads), router_smem_bytes(a.E), st, false, a);
}

// The grouped kernels with 4 tokens per pass have 7 consumer warps, one
// 32-chunk column block of a row each: rows of at most 7 x 32 x 32 = 7168
// values.  A wider hidden or FFN row takes the one-token-per-pass variants
// (16 and 8 consumer warps, rows up to 8192), which loop over an expert's
// tokens for any batch.
static bool grouped_one(const LayerArgs& a) {
  constexpr int kWide = 7 * 32 * 32;
  return a.T == 1 || a.H > kWide || std::max(a.F, a.Fs) > kWide;
}

static cudaError_t launch_experts_g(LayerArgs& a, int num_sms, cudaStream_t st, bool pdl) {
  const bool one = grouped_one(a);
  cudaError_t e;
  if (one)
    e = launch_ex((const void*)gateup_kernel<1, 16>, dim3(num_sms), dim3(17 * 32),
                  gateup_smem_bytes(a, 1, 16), st, pdl, a);
  else
    e = launch_ex((const void*)gateup_kernel<4, 7>, dim3(num_sms), dim3(8 * 32),
                  gateup_smem_bytes(a, 4, 7), st, pdl, a);
  if (e || (e = mark(a, 2, st))) return e;
  if (one)
    e = launch_ex((const void*)down_kernel<1, 8>, dim3(num_sms), dim3(9 * 32),
                  down_smem_bytes(a, 1, 8), st, pdl, a);
  else
    e = launch_ex((const void*)down_kernel<4, 7>, dim3(num_sms), dim3(8 * 32),
                  down_smem_bytes(a, 4, 7), st, pdl, a);
  return e;
}

// The router alone, then (after the expert cache is updated) everything
// else: the general path's split for the expert cache.
cudaError_t launch_decode_router(const LayerArgs& a, int num_sms, cudaStream_t st) {
  return launch_router_g(a, num_sms, st);
}

cudaError_t launch_decode_experts(const LayerArgs& in, int num_sms, cudaStream_t st) {
  LayerArgs a = in;
  const bool one = grouped_one(a);
  plan_decode(a, num_sms, one ? 16 : 7, one ? 8 : 7, one ? 1 : 4);
  return launch_experts_g(a, num_sms, st, false);
}

cudaError_t launch_decode(const LayerArgs& in, int num_sms, cudaStream_t st) {
  LayerArgs a = in;
  const bool one = grouped_one(a);
  const bool pdl = !a.prof_on;
  plan_decode(a, num_sms, one ? 16 : 7, one ? 8 : 7, one ? 1 : 4);
  cudaError_t e;
  if ((e = mark(a, 0, st))) return e;
  e = launch_router_g(a, num_sms, st);
  if (e || (e = mark(a, 1, st))) return e;
  if ((e = launch_experts_g(a, num_sms, st, pdl))) return e;
  return mark(a, 3, st);
}

}  // namespace moe
