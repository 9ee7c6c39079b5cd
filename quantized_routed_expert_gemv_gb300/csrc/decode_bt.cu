// decode_bt.cu -- decode of a few tokens (2 <= B <= 16) with every selected
// expert's weights read once per step.
//
// TurboFieldfare page, section "Token üretim süreci": one fetched expert
// serves all the rows routed to it.  For a small batch over many experts
// most experts serve one token and the shared expert serves all of them, so
// the step is the single-token step's weight stream (the fused kernel of
// decode_b1.cu) with a short token loop per item:
//
// router_kernel    (decode.cu) logits, top-k and the grouping by expert;
//                  CTAs of its own (after the logits CTAs) write every
//                  token's activations in the fixed-point chunk form of
//                  gemv.cuh once, and count themselves done on a control word.
// ffn_bt_kernel    one persistent kernel over one claimed item list:
//                  gate|up items (rth gate + rth up rows of one expert) and
//                  down items (RTD rows of H of one expert's down matrix),
//                    G(0) .. G(n - 1) D(0) .. D(n - 1)    (entry 0: shared)
//                  as in the single-token kernel.  A stage holds weights
//                  only; the consumer threads loop over the item's tokens,
//                  reading each token's fixed-point activations (gate|up) or
//                  its fixed-point h group (down) from L2, so each weight
//                  byte is read from HBM once and applied to every token of
//                  its expert.  Epilogue warps gather the per-token row sums:
//                  SwiGLU + fixed-point h groups per (expert, token) pair for
//                  gate|up items, weighted rows per pair for down items.
// combine_bt_kernel out[t] = y_shared[t] + sum over t's ranks i of the pair's
//                  weighted rows, in that fixed order, so outputs do not
//                  depend on which CTA did which item.
#include <algorithm>

#include "common.cuh"
#include "fused.cuh"
#include "gemv.cuh"
#include "kernels.h"

namespace moe {

constexpr int kBtWarps = 16;                     // consumer warps
constexpr int kBtThreads = (kBtWarps + 3) * 32;  // + producer + two epilogue warps
constexpr int kBtMaxStages = 8;
constexpr int kBtCombineThreads = 256;
constexpr int kBtVals = 8;  // values an epilogue lane gathers before the stage is released

struct BtEnt {         // one expert entry of the step, as the producer and the consumers use it
  const uint8_t* rec;  // record base
  int pair0;           // its first (entry, token) pair
  int ntok;            // tokens routed to it
};

struct BtSmem {
  int wsum, code, ent, tok, bars, total;
};

// Dynamic shared memory: NST stages, then per stage the consumer warps' row
// sums [NT tokens][kBtWarps][8], the stages' item codes (+ the step's entry
// count), the entry table [n_ent_max] and the token of every pair [np_max].
__host__ __device__ inline BtSmem bt_smem(int nst, int stage, int nt, int n_ent_max, int np_max) {
  BtSmem s;
  s.wsum = nst * stage;
  s.code = s.wsum + nst * nt * kBtWarps * 8 * 4;
  s.ent = s.code + (kBtMaxStages + 4) * 4;
  s.tok = s.ent + n_ent_max * static_cast<int>(sizeof(BtEnt));
  s.bars = (s.tok + np_max + 15) / 16 * 16;
  s.total = s.bars + 3 * nst * 8 + 16;  // full, empty, partial sums done
  return s;
}

// Pairs: the shared expert's token t is pair t (t < nsh = B when there is a
// shared expert); the router's grouped pair position q is pair nsh + q.
// Pair P's fixed-point h block (96 bytes per 32-value chunk) starts at byte
// bt_hoff(P) of the workspace's h area: shared blocks first, then routed
// ones, each padded to whole 128-byte lines.
__host__ __device__ inline size_t bt_hblock(int Fe) { return (static_cast<size_t>(3 * Fe) + 127) / 128 * 128; }
__device__ __forceinline__ size_t bt_hoff(int P, int nsh, int Fs, int F) {
  return P < nsh ? P * bt_hblock(Fs) : nsh * bt_hblock(Fs) + (P - nsh) * bt_hblock(F);
}



// Routing weight of pair P (1 for the shared expert's pairs).
__device__ __forceinline__ float bt_weight(const LayerArgs& a, int P, int nsh) {
  if (P < nsh) return 1.f;
  int q = __ldcg(a.ws.pair_slot + (P - nsh));
  q = min(max(q, 0), a.T * a.k - 1);
  return __ldcg(a.weights + q);
}

template <int R, int NT>  // R: gate|up rows per thread per item (R/2 gate + R/2 up); NT: tokens per item
__global__ void __launch_bounds__(kBtThreads, 1) ffn_bt_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NCW = kBtWarps;
  const int H = a.H, C = H >> 5, WC = (C + 31) >> 5, NRL = a.gu_nrl, NAW = NRL * WC;
  constexpr int RH = R / 2;
  const int rth = RH * NRL;
  const int T = a.T, NST = a.f1_nst, SB = a.f1_stage, RTD = a.f1_rt;
  const int has_sh = a.Fs > 0 ? 1 : 0, nsh = has_sh * T;
  const int n_ent_max = has_sh + min(a.E, T * a.k), np_max = nsh + T * a.k;
  const BtSmem L = bt_smem(NST, SB, NT, n_ent_max, np_max);
  float* wsum = reinterpret_cast<float*>(smem + L.wsum);
  volatile int* s_code = reinterpret_cast<volatile int*>(smem + L.code);
  volatile int* s_nent = s_code + kBtMaxStages;
  BtEnt* tab = reinterpret_cast<BtEnt*>(smem + L.ent);
  uint8_t* s_tok = smem + L.tok;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + NST;   // consumers and the position's epilogue warp are done
  uint64_t* pdone = empty + NST;  // every consumer's row sums of the position are in
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&full[s], 1), mbar_init(&empty[s], NCW + 1), mbar_init(&pdone[s], NCW);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int tiles_s = has_sh ? a.Fs / rth : 0, tiles_r = a.F / rth, ndn = H / RTD;
  const int n_pre = tiles_s;  // items that need no routing: the shared gate|up

  if (warp == NCW) {  // ---------------- producer warp (lane 0 issues; the warp builds the tables)
    const uint64_t pol = policy_evict_first();
    unsigned* claim = &a.ws.ctl[2];
    const F1Div dr = f1_div(tiles_r), dn = f1_div(ndn);
    int it = 0, n_items = n_pre, n_ent = has_sh, checked = -1, cur = 0, nxt = 0;
    bool ok = true;
    RingPos pos;
    if (has_sh) {  // the shared expert needs no routing: entry 0, pairs 0 .. T-1
      if (lane == 0) {
        BtEnt t;
        t.rec = a.shared, t.pair0 = 0, t.ntok = T;
        tab[0] = t;
      }
      for (int t = lane; t < T; t += 32) s_tok[t] = static_cast<uint8_t>(t);
      __syncwarp();
    }
    if (lane == 0) {
      cur = static_cast<int>(atomicAdd(claim, 1u));
      nxt = static_cast<int>(atomicAdd(claim, 1u));
    }
    for (int phase = 0; phase < 2 && ok; ++phase) {
      if (phase == 1) {
        // routed items: wait for the router, then the warp looks the step's
        // experts and pairs up once into shared memory
        pdl_wait();
        const int n_act = min(clamp_n_act(a), n_ent_max - has_sh);
        const int npr = T * a.k;
        for (int j = lane; j < n_act; j += 32) {
          const B1Entry en = b1_entry(a, has_sh + j, has_sh);
          if (a.slot_tag && a.slot_tag[en.slot] != en.expert) latch_error(&a.ws.ctl[0], kErrResidency);
          int q0 = a.ws.act_off[j], cnt = a.ws.act_cnt[j];
          if (q0 < 0 || q0 >= npr || cnt < 1 || cnt > min(NT, npr - q0)) {  // not from a correct router
            latch_error(&a.ws.ctl[0], kErrRange);
            q0 = min(max(q0, 0), npr - 1), cnt = min(max(cnt, 1), min(NT, npr - q0));
          }
          BtEnt t;
          t.rec = en.rec, t.pair0 = nsh + q0, t.ntok = cnt;
          tab[has_sh + j] = t;
        }
        for (int q = lane; q < npr; q += 32) {
          int tk = a.ws.pair_token[q];
          if (tk < 0 || tk >= T) latch_error(&a.ws.ctl[0], kErrRange), tk = 0;
          s_tok[nsh + q] = static_cast<uint8_t>(tk);
        }
        __syncwarp();
        n_items = n_pre + n_act * tiles_r + (has_sh + n_act) * ndn;
        n_ent = has_sh + n_act;
        if (lane == 0) *s_nent = n_ent;
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
          const uint8_t* rec = tab[e].rec;
          if (!gate && e != checked) {  // the expert's h must be complete before its down items
            if (!wait_count(&a.ws.hcnt[e], sh ? tiles_s : tiles_r)) {
              latch_error(&a.ws.ctl[0], kErrTimeout);
              ok = false;
              break;
            }
            checked = e;
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
            bulk_g2s(st, rec + off.gate_codes + j0 * (H / 2), cb, &full[s], pol);
            bulk_g2s(st + cb, rec + off.up_codes + j0 * (H / 2), cb, &full[s], pol);
            bulk_g2s(st + 2 * cb, rec + off.gate_sb + j0 * (H / 16), sbb, &full[s], pol);
            bulk_g2s(st + 2 * cb + sbb, rec + off.up_sb + j0 * (H / 16), sbb, &full[s], pol);
          } else {
            const int Fe = sh ? a.Fs : a.F;
            const uint32_t cb = RTD * (Fe / 2), sbb = RTD * (Fe / 16);
            const size_t r0 = static_cast<size_t>(tile) * RTD;
            mbar_arrive_expect_tx(&full[s], cb + sbb);
            bulk_g2s(st, rec + off.down_codes + r0 * (Fe / 2), cb, &full[s], pol);
            bulk_g2s(st + cb, rec + off.down_sb + r0 * (Fe / 16), sbb, &full[s], pol);
          }
        }
      }
      ok = __shfl_sync(kAll, ok ? 1 : 0, 0) != 0;
    }
    // The grid completes after the router's, even when a wait gave up before
    // the routed items: the combine, which clears the router's conversion
    // count, relies on it.
    pdl_wait();
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
    for (int it = q;; it += 2) {
      const int s = it % NST;
      const uint32_t ph = (it / NST) & 1;
      if (!mbar_wait_sleep_warp(&full[s], ph)) {
        if (lane == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
        break;
      }
      const int code = s_code[s];
      if (code < 0) break;
      const int gate = code & 1, e = code >> 20, tile = (code >> 1) & 0x7FFFF;
      const bool sh_row = has_sh && e == 0;
      const BtEnt en = tab[e];
      const int ntok = min(en.ntok, NT);
      const float* ws0 = wsum + static_cast<size_t>(s) * NT * NCW * 8;
      // Lane u < ntok holds the routing weight of the item's pair u, loaded
      // before the wait for the consumers' sums so its latency is hidden.
      const float pw = (!gate && lane < ntok) ? bt_weight(a, en.pair0 + lane, nsh) : 1.f;
      if (!mbar_wait_sleep_warp(&pdone[s], ph)) {
        if (lane == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
        break;
      }
      // The values of the item (pair u, row) are gathered from the stage's
      // row sums kBtVals per lane at a time; the stage is released as soon
      // as the last round is gathered, and the stores follow.
      const int rows = gate ? rth : RTD, nv = ntok * rows;
      const D1Geo& g = sh_row ? gs : gr;
      for (int r0 = 0; r0 < nv; r0 += 32 * kBtVals) {
        float val[kBtVals];
#pragma unroll
        for (int i = 0; i < kBtVals; ++i) {
          const int v = r0 + i * 32 + lane;
          val[i] = 0.f;
          if (v < nv) {
            const int u = v / rows, r = v - u * rows;
            if (gate) {
              // SwiGLU of the gathered gate and up sums of row r
              const int rlj = r / RH, mj = r % RH;
              float gg = 0.f, up = 0.f;
              for (int w = 0; w < WC; ++w) {
                const float* p = ws0 + (u * NCW + rlj * WC + w) * 8;
                gg += p[mj];
                up += p[RH + mj];
              }
              val[i] = silu1(gg) * up;
            } else {
              const int rl = r % g.NRL, m = r / g.NRL;
              float y = 0.f;
              for (int w = 0; w < g.WC; ++w) y += ws0[(u * NCW + rl * g.WC + w) * 8 + m];
              val[i] = y;
            }
          }
        }
        __syncwarp();
        if (r0 + 32 * kBtVals >= nv && lane == 0) mbar_arrive(&empty[s]);  // the stage is free
#pragma unroll
        for (int i = 0; i < kBtVals; ++i) {
          const int v0 = r0 + i * 32;
          if (v0 >= nv) break;  // the same on every lane
          const int v = v0 + lane;
          const bool act = v < nv;
          const int u = act ? v / rows : 0, r = act ? v - u * rows : 0;
          if (gate) {
            // fixed-point h groups (rth is a multiple of 8, so an 8-lane
            // segment is one group of one pair)
            publish_hgroup_at(a.ws.hx + bt_hoff(en.pair0 + u, nsh, a.Fs, a.F), (sh_row ? a.Fs : a.F) >> 5,
                              tile * rth + r, val[i], act, lane);
          } else {
            const float p = __shfl_sync(kAll, pw, u);
            if (act)
              a.ws.ypart[static_cast<size_t>(en.pair0 + u) * H + static_cast<size_t>(tile) * RTD + r] = p * val[i];
          }
        }
      }
      if (gate) {
        __syncwarp();
        if (lane == 0) red_add_release_gpu(&a.ws.hcnt[e], 1u);
      }
    }
    return;
  }

  // ---------------------------------------------------- consumers
  const int rl = warp / WC, wc = warp % WC, col = wc * 32 + lane;
  const bool gact = warp < NAW && col < C;  // this lane's column of a gate|up item
  const D1Geo gs = d1_geo(has_sh ? a.Fs : a.F, warp, lane), gr = d1_geo(a.F, warp, lane);
  // the router's fixed-point activations: words [T][4][C] uint4, then [T][C]
  // (2^e, plain sum of the chunk), read from L2 like the h blocks
  const uint4* xqw = reinterpret_cast<const uint4*>(a.ws.xq);
  const float2* xqs = reinterpret_cast<const float2*>(a.ws.xq + static_cast<size_t>(T) * C * 64);
  bool xready = false, abort = false;
  // Token t's activations of this lane's column into L1 ahead of their use.
  // The router writes them before it counts itself done and they do not
  // change for the rest of the grid, so once the count has been acquired
  // they are read through L1 (one token's 72 bytes a column fit beside the
  // next one's prefetch).  Only for rows of at least 4096 values: there
  // the L2 round trip at the start of a token's pass is the larger cost
  // (H = 7168, B = 4: 302 -> 295 us per step); at H = 2048 the added
  // instructions cost more than they hide (B = 4 and 16: 2-4% slower).
  const bool xpf = C >= 128;
  const auto prefetch_x = [&](int t) {
    if (!xpf || !gact || !xready) return;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      asm volatile("prefetch.global.L1 [%0];" ::"l"(xqw + (static_cast<size_t>(t) * 4 + k) * C + col));
    asm volatile("prefetch.global.L1 [%0];" ::"l"(xqs + static_cast<size_t>(t) * C + col));
  };
  // The next ring position's first token, when its weights are already in
  // and it is a gate|up item.
  const auto prefetch_next = [&](const RingPos& at) {
    if (!xpf) return;
    RingPos nx = at;
    nx.next(NST);
    if (!mbar_test_wait(&full[nx.s], nx.ph)) return;
    const int c2 = s_code[nx.s];
    if (c2 < 0 || !(c2 & 1)) return;
    prefetch_x(s_tok[tab[c2 >> 20].pair0]);
  };

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
    const int e = code >> 20;
    const BtEnt en = tab[e];
    const int ntok = min(en.ntok, NT);
    float* ws0 = wsum + static_cast<size_t>(s) * NT * NCW * 8;
    if (code & 1) {  // gate|up item
      if (!xready && !abort) {
        // the router's CTAs that convert the tokens count themselves done
        xready = __all_sync(kAll, wait_count(&a.ws.ctl[10], static_cast<unsigned>(a.xq_nconv))) != 0;
        if (!xready) {
          if (lane == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
          abort = true;
        }
      }
      const uint8_t* stsb = st + 2 * rth * (H / 2);
      for (int u = 0; u < ntok; ++u) {
        const int t = s_tok[en.pair0 + u];
        float part[R];
#pragma unroll
        for (int m = 0; m < R; ++m) part[m] = 0.f;
        if (gact && !abort) {
          XChunk X;
          const uint4 k0 = __ldca(xqw + (static_cast<size_t>(t) * 4 + 0) * C + col);
          const uint4 k1 = __ldca(xqw + (static_cast<size_t>(t) * 4 + 1) * C + col);
          const uint4 k2 = __ldca(xqw + (static_cast<size_t>(t) * 4 + 2) * C + col);
          const uint4 k3 = __ldca(xqw + (static_cast<size_t>(t) * 4 + 3) * C + col);
          const float2 ss = __ldca(xqs + static_cast<size_t>(t) * C + col);
          if (u + 1 < ntok) prefetch_x(s_tok[en.pair0 + u + 1]);
          else prefetch_next(pos);
          X.eh[0] = k0.x, X.eh[1] = k0.y, X.eh[2] = k0.z, X.eh[3] = k0.w;
          X.el[0] = k1.x, X.el[1] = k1.y, X.el[2] = k1.z, X.el[3] = k1.w;
          X.oh[0] = k2.x, X.oh[1] = k2.y, X.oh[2] = k2.z, X.oh[3] = k2.w;
          X.ol[0] = k3.x, X.ol[1] = k3.y, X.ol[2] = k3.z, X.ol[3] = k3.w;
#pragma unroll
          for (int m = 0; m < R; ++m) {
            const int r = (m < RH) ? (RH * rl + m) : (rth + RH * rl + m - RH);
            const uint4 qv = *reinterpret_cast<const uint4*>(st + r * (H / 2) + col * 16);
            const uint32_t sbw = *reinterpret_cast<const uint32_t*>(stsb + r * (H / 16) + (col >> 1) * 4);
            part[m] = fmaf(bf16lo(sbw) * ss.x, static_cast<float>(dot_chunk(qv, X)), bf16hi(sbw) * ss.y);
          }
        }
        constexpr int LPR = 32 / R;  // lanes per row after the butterfly
        float v;
        if constexpr (R == 8) v = bfly8(part, lane);
        else v = bfly4b(part, lane);
        if ((lane & (LPR - 1)) == 0) ws0[(u * NCW + warp) * 8 + lane / LPR] = v;
      }
    } else {  // down item: RTD rows of one expert, each pair's h group from L2
      const bool sh = has_sh && e == 0;
      const D1Geo& g = sh ? gs : gr;
      const int Fe = sh ? a.Fs : a.F, nc = Fe >> 5, rowb = Fe / 2, sbrow = Fe / 16;
      const int RR = RTD / g.NRL;  // rows per thread
      const uint8_t* stsb = st + RTD * rowb;
      for (int u = 0; u < ntok; ++u) {
        float part[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) part[m] = 0.f;
        if (g.act) {
          const uint8_t* xb = a.ws.hx + bt_hoff(en.pair0 + u, nsh, a.Fs, a.F);
          const uint4* xw = reinterpret_cast<const uint4*>(xb);
          XChunk Xh;
          const uint4 g0 = __ldcg(xw + 0 * nc + g.col), g1 = __ldcg(xw + 1 * nc + g.col),
                      g2 = __ldcg(xw + 2 * nc + g.col), g3 = __ldcg(xw + 3 * nc + g.col);
          const float4 sc4 = __ldcg(reinterpret_cast<const float4*>(xb + 64 * nc) + g.col);
          const float4 sm4 = __ldcg(reinterpret_cast<const float4*>(xb + 80 * nc) + g.col);
          if (u + 1 == ntok) prefetch_next(pos);
          Xh.eh[0] = g0.x, Xh.eh[1] = g0.y, Xh.eh[2] = g0.z, Xh.eh[3] = g0.w;
          Xh.el[0] = g1.x, Xh.el[1] = g1.y, Xh.el[2] = g1.z, Xh.el[3] = g1.w;
          Xh.oh[0] = g2.x, Xh.oh[1] = g2.y, Xh.oh[2] = g2.z, Xh.oh[3] = g2.w;
          Xh.ol[0] = g3.x, Xh.ol[1] = g3.y, Xh.ol[2] = g3.z, Xh.ol[3] = g3.w;
          const float scp[4] = {sc4.x, sc4.y, sc4.z, sc4.w};
          const float psx = (sm4.x + sm4.y) + (sm4.z + sm4.w);
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
        if ((lane & 3) == 0) ws0[(u * NCW + warp) * 8 + (lane >> 2)] = v;
      }
    }
    __syncwarp();  // the lanes' sums before lane 0's arrivals (release at CTA scope)
    if (lane == 0) mbar_arrive(&pdone[s]), mbar_arrive(&empty[s]);
  }
}

// out[t][r] = y_shared[t][r] + sum_i ypart[pair of (t, rank i)][r], ranks in
// order; also clears the control word the router's conversion CTAs count on
// (every reader of it belonged to the finished ffn_bt grid).
__global__ void __launch_bounds__(kBtCombineThreads) combine_bt_kernel(const __grid_constant__ LayerArgs a) {
  __shared__ int inv[kBtMaxTokens * kMaxTopK];  // (token, rank) -> grouped pair position
  const int T = a.T, k = a.k, H = a.H, nsh = a.Fs > 0 ? T : 0, npr = T * k;
  pdl_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0) a.ws.ctl[10] = 0u;
  for (int q = threadIdx.x; q < npr; q += blockDim.x) inv[q] = 0;
  __syncthreads();
  for (int q = threadIdx.x; q < npr; q += blockDim.x) {
    const int slot = __ldcg(a.ws.pair_slot + q);
    if (slot >= 0 && slot < npr) inv[slot] = q;
  }
  __syncthreads();
  const size_t n = static_cast<size_t>(T) * H;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / H), r = static_cast<int>(i - static_cast<size_t>(t) * H);
    float out = nsh ? __ldcg(a.ws.ypart + static_cast<size_t>(t) * H + r) : 0.f;
    for (int j = 0; j < k; ++j)
      out += __ldcg(a.ws.ypart + static_cast<size_t>(nsh + inv[t * k + j]) * H + r);
    a.out_bf16[i] = f32_to_bf16_rne(out);
    if (a.out_f32) a.out_f32[i] = out;
  }
}

// ============================================================================
// Host side.
// ============================================================================

size_t bt_smem_bytes(const LayerArgs& a, int nt) {
  const int has_sh = a.Fs > 0 ? 1 : 0;
  return bt_smem(a.f1_nst, a.f1_stage, nt, has_sh + std::min(a.E, a.T * a.k), has_sh * a.T + a.T * a.k).total;
}

static int bt_nt(int T) { return T <= 4 ? 4 : kBtMaxTokens; }

// Row-lanes of the down mapping for an h row of width Fe (as d1_geo).
static int bt_nrl(int Fe) {
  const int C = Fe / 32, WC = (C + 31) / 32;
  int n = kD1Warps / WC;
  while (n & (n - 1)) n &= n - 1;
  return std::max(1, n);
}

// Geometry of the few-token kernel for a.T tokens: gate|up items of R rows
// per thread (8, else 4), down items of RTD rows (a divisor of H, a multiple
// of 4 and of both widths' row-lanes, at most 8 rows per thread), and the
// deepest ring the shared memory holds.  Takes the largest items that keep a
// ring of three stages (a ring of two leaves one stage of copies in flight
// per SM, too little to cover HBM latency at this SM's share of the
// bandwidth); a ring of two only when no plan keeps three.  False when no
// plan keeps two stages.
bool plan_bt(LayerArgs& a, int num_sms, int smem_optin) {
  (void)num_sms;
  if (a.T < 2 || a.T > kBtMaxTokens) return false;
  const int H = a.H, C = H / 32, WC = (C + 31) / 32;
  int nrl = std::max(1, kBtWarps / WC);
  while (nrl & (nrl - 1)) nrl &= nrl - 1;
  const int Fm = std::max(a.F, a.Fs), nr = bt_nrl(a.F), ns = a.Fs ? bt_nrl(a.Fs) : nr;
  const int nt = bt_nt(a.T), has_sh = a.Fs > 0 ? 1 : 0;
  const int budget = smem_optin - 1024;
  int fb_R = 0, fb_rt = 0, fb_sb = 0, fb_nst = 0;  // the first two-stage plan
  for (int R = 8; R >= 4; R -= 4) {
    const int rth = (R / 2) * nrl;
    if (rth % 8 || rth > 64 || a.F % rth || (a.Fs && a.Fs % rth)) continue;
    const int gst = 2 * rth * (H / 2 + H / 16);
    for (int rt = 64; rt >= 4; --rt) {
      if (H % rt || rt % 4 || rt % nr || rt % ns || rt / nr > 8 || rt / ns > 8) continue;
      if (H / rt > kMaxDim / 8) break;
      const int sb = (std::max(gst, rt * (Fm / 2 + Fm / 16)) + 127) / 128 * 128;
      const int fixed = bt_smem(0, sb, nt, has_sh + std::min(a.E, a.T * a.k), has_sh * a.T + a.T * a.k).total;
      const int per = bt_smem(1, sb, nt, 0, 0).total - bt_smem(0, sb, nt, 0, 0).total;
      const int nst = std::min(kBtMaxStages, (budget - fixed) / per);
      if (nst >= 3) {
        a.gu_nrl = nrl, a.gu_rows = R, a.f1_rt = rt, a.f1_stage = sb, a.f1_nst = nst;
        return true;
      }
      if (nst == 2 && fb_nst == 0) fb_R = R, fb_rt = rt, fb_sb = sb, fb_nst = 2;
    }
  }
  if (fb_nst < 2) return false;
  a.gu_nrl = nrl, a.gu_rows = fb_R, a.f1_rt = fb_rt, a.f1_stage = fb_sb, a.f1_nst = fb_nst;
  return true;
}

cudaError_t set_bt_attributes(int smem_optin) {
  const void* fns[] = {(const void*)ffn_bt_kernel<4, 4>, (const void*)ffn_bt_kernel<4, kBtMaxTokens>,
                       (const void*)ffn_bt_kernel<8, 4>, (const void*)ffn_bt_kernel<8, kBtMaxTokens>};
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

static cudaError_t launch_bt(const void* fn, int grid, int block, size_t smem, cudaStream_t st, bool pdl,
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

static cudaError_t mark_bt(const LayerArgs& a, int i, cudaStream_t st) {
  return a.prof_on ? cudaEventRecord(static_cast<cudaEvent_t>(a.prof[i]), st) : cudaSuccess;
}

int decode_router_grid(const LayerArgs& a, int num_sms);
cudaError_t launch_decode_router(const LayerArgs& a, int num_sms, cudaStream_t st);

// Number of router CTAs that convert the tokens to fixed point (launched
// after the logits CTAs).
int bt_nconv(const LayerArgs& a, int num_sms) {
  const int chunks = a.T * (a.H / 32);
  return std::max(1, std::min(decode_router_grid(a, num_sms), (chunks + 511) / 512));
}

// The router (with the tokens' fixed-point conversion), the fused kernel and
// the combine; `a` planned by plan_bt.  Profile events: before the router,
// before the fused kernel, before the combine, after it.
cudaError_t launch_decode_bt(const LayerArgs& in, int num_sms, cudaStream_t st) {
  LayerArgs a = in;
  a.xq_nconv = bt_nconv(a, num_sms);
  const bool pdl = !a.prof_on;
  const int nt = bt_nt(a.T);
  const void* fn = a.gu_rows == 8 ? (nt == 4 ? (const void*)ffn_bt_kernel<8, 4> : (const void*)ffn_bt_kernel<8, kBtMaxTokens>)
                                  : (nt == 4 ? (const void*)ffn_bt_kernel<4, 4> : (const void*)ffn_bt_kernel<4, kBtMaxTokens>);
  const int cgrid = std::max(1, std::min(num_sms, (a.T * a.H + kBtCombineThreads - 1) / kBtCombineThreads));
  cudaError_t e;
  if ((e = mark_bt(a, 0, st)) || (e = launch_decode_router(a, num_sms, st)) || (e = mark_bt(a, 1, st)) ||
      (e = launch_bt(fn, num_sms, kBtThreads, bt_smem_bytes(a, nt), st, pdl, a)) || (e = mark_bt(a, 2, st)) ||
      (e = launch_bt((const void*)combine_bt_kernel, cgrid, kBtCombineThreads, 0, st, pdl, a)))
    return e;
  return mark_bt(a, 3, st);
}

}  // namespace moe
