// fused.cuh -- device helpers of the persistent fused decode kernels
// (decode_b1.cu: one token; decode_bt.cu: a few tokens, each expert's
// weights read once): warp reductions of per-lane row partials, the
// fixed-point h groups that gate|up items publish for the down items, the
// step's expert entries, and the claimed item list.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "gemv.cuh"
#include "kernels.h"

namespace moe {

constexpr int kD1Warps = 16;  // consumer warps of the down mapping (d1_geo)

namespace {

constexpr unsigned kAll = kFull;

__device__ __forceinline__ float warp_add(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kAll, v, o);
  return v;
}

// Sums eight per-lane row partials over the warp; lane L ends with the total
// of row L >> 2.
__device__ __forceinline__ float bfly8(const float (&p)[8], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float k[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b4 ? p[4 + i] : p[i], send = b4 ? p[i] : p[4 + i];
    k[i] = keep + __shfl_xor_sync(kAll, send, 16);
  }
  float k2[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b3 ? k[2 + i] : k[i], send = b3 ? k[i] : k[2 + i];
    k2[i] = keep + __shfl_xor_sync(kAll, send, 8);
  }
  float v = b2 ? k2[1] : k2[0];
  const float send = b2 ? k2[0] : k2[1];
  v += __shfl_xor_sync(kAll, send, 4);
  v += __shfl_xor_sync(kAll, v, 2);
  v += __shfl_xor_sync(kAll, v, 1);
  return v;
}

// Four-row version: lane L ends with the total of row 2*bit4 + bit3.
__device__ __forceinline__ float bfly4b(const float (&p)[4], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8;
  float k[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b4 ? p[2 + i] : p[i], send = b4 ? p[i] : p[2 + i];
    k[i] = keep + __shfl_xor_sync(kAll, send, 16);
  }
  float v = b3 ? k[1] : k[0];
  const float send = b3 ? k[0] : k[1];
  v += __shfl_xor_sync(kAll, send, 8);
  v += __shfl_xor_sync(kAll, v, 4);
  v += __shfl_xor_sync(kAll, v, 2);
  v += __shfl_xor_sync(kAll, v, 1);
  return v;
}

__device__ __forceinline__ float silu1(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ int clamp_n_act(const LayerArgs& a) {
  const int n = *reinterpret_cast<volatile int*>(a.ws.n_act);
  return n < 0 ? 0 : (n > a.E ? a.E : n);
}

struct B1Entry {
  const uint8_t* rec;
  const RecordOffsets* off;
  int Fe, pair, shared, expert, slot;
};

__device__ __forceinline__ B1Entry b1_entry(const LayerArgs& a, int idx, int has_sh) {
  B1Entry en;
  if (has_sh && idx == 0) {
    en.rec = a.shared, en.off = &a.off_s, en.Fe = a.Fs, en.pair = 0, en.shared = 1, en.expert = -1, en.slot = -1;
    return en;
  }
  const int i = idx - has_sh;
  int e = a.ws.act_expert[i];
  if (e < 0 || e >= a.E) e = 0;
  int slot = e;
  if (a.slot_of) {  // residency: a slot outside the pool is never read
    slot = a.slot_of[e];
    if (slot < 0 || slot >= a.n_slots) latch_error(&a.ws.ctl[0], kErrResidency), slot = 0;
  }
  en.rec = a.records + static_cast<size_t>(slot) * a.off_r.stride;
  en.off = &a.off_r, en.Fe = a.F, en.pair = a.ws.act_off[i], en.shared = 0, en.expert = e;
  en.slot = slot;
  return en;
}


// Writes the fixed-point form of one 8-value group of an h row.  The warp's
// 8-lane segments hold groups: lane 8g + p holds element f (f = 8 * (group)
// + p) of the row with value v (0 where `act` is false).  The row's chunks
// start at chunk c0 and number nc; its block of 96 * nc bytes starts at byte
// 96 * c0 of hx, so the down kernels copy it in one piece.  In the block:
// the word of kind K (0: high bytes of the even elements, 1: their low
// bytes, 2 and 3: the same for the odd elements) of group i of chunk c sits
// at 32-bit word (K * nc + c) * 4 + i; the group's 2^e at float
// 16 * nc + c * 4 + i and its plain sum at float 20 * nc + c * 4 + i.
// publish_hgroup into the block that starts at blk_base (the chunk layout
// above, any 16-byte aligned start).
__device__ __forceinline__ void publish_hgroup_at(uint8_t* blk_base, int nc, int f, float v, bool act, int lane) {
  float amax = fabsf(v), sum = v;
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, o));
    sum += __shfl_xor_sync(kAll, sum, o);
  }
  // 2^e with amax / 2^e < 2^15 and its inverse, straight from amax's
  // exponent field (the same 2^e as fixed_scale for amax >= 2^-112; below
  // that, 2^-126, which keeps |v| / 2^e < 2^15)
  const int eb = max(static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu), 15);
  const float scale = __uint_as_float(static_cast<uint32_t>(eb - 14) << 23);
  const float inv = __uint_as_float(static_cast<uint32_t>(268 - eb) << 23);
  const int X = min(max(__float2int_rn(v * inv), -32767), 32767);
  // lane p < 4 of the segment builds the word of kind p from elements
  // par + 2b (b = 0..3) of the group, par = p >> 1
  const int base = lane & ~7, p = lane & 7, par = (p >> 1) & 1, hi = (p & 1) == 0;
  int byte[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int xv = __shfl_sync(kAll, X, base + par + 2 * b);
    byte[b] = hi ? (xv >> 8) : xv;
  }
  if (act && p < 4) {
    const int c = f >> 5, i = (f >> 3) & 3;
    uint32_t* blk = reinterpret_cast<uint32_t*>(blk_base);
    blk[(p * nc + c) * 4 + i] = pack4(byte[0], byte[1], byte[2], byte[3]);
    if (p == 0) {
      float* f = reinterpret_cast<float*>(blk);
      f[16 * nc + c * 4 + i] = scale;
      f[20 * nc + c * 4 + i] = sum;
    }
  }
}

__device__ __forceinline__ void publish_hgroup(const LayerArgs& a, int c0, int nc, int f, float v, bool act,
                                               int lane) {
  publish_hgroup_at(a.ws.hx + static_cast<size_t>(c0) * 96, nc, f, v, act, lane);
}

struct D1Geo {  // thread mapping for one expert width
  int C, WC, NRL, rl, col;
  bool act;
};

__device__ __forceinline__ D1Geo d1_geo(int Fe, int warp, int lane) {
  D1Geo g;
  g.C = Fe >> 5;
  g.WC = (g.C + 31) >> 5;
  int n = kD1Warps / g.WC;
  while (n & (n - 1)) n &= n - 1;
  g.NRL = n;
  g.rl = warp / g.WC;
  g.col = (warp % g.WC) * 32 + lane;
  g.act = g.rl < g.NRL && g.col < g.C;
  return g;
}

// n / d for n * d < 2^40 as one 64-bit multiply: m = ceil(2^40 / d).
struct F1Div {
  unsigned long long m;
  int d;
};
__device__ __forceinline__ F1Div f1_div(int d) {
  F1Div r;
  r.d = d;
  r.m = ((1ull << 40) + static_cast<unsigned long long>(d) - 1) / static_cast<unsigned long long>(d);
  return r;
}
__device__ __forceinline__ int f1_q(int n, const F1Div& v) {
  return static_cast<int>((static_cast<unsigned long long>(n) * v.m) >> 40);
}

// Item code in shared memory: entry << 20 | tile << 1 | gate (-1: end).
__device__ __forceinline__ int f1_code(int gate, int entry, int tile) { return (entry << 20) | (tile << 1) | gate; }

// Claim index -> (gate, entry, tile) for the n_ent experts of the step
// (entry 0 the shared expert when there is one, its gate|up block tiles_s
// items; every other gate|up block tiles_r items, every down block ndn
// items): every gate|up item, expert by expert, then every down item.  Only
// the shared expert's gate|up comes before the router's output is needed.
// The divisions use the reciprocals dr (tiles_r) and dn (ndn).
__device__ __forceinline__ int f1_item(int i, int has_sh, int tiles_s, int n_ent, const F1Div& dr,
                                       const F1Div& dn) {
  const int tiles_r = dr.d, ndn = dn.d;
  const int g0 = has_sh ? tiles_s : tiles_r;
  if (i < g0) return f1_code(1, 0, i);
  const int gates = g0 + (n_ent - 1) * tiles_r;
  if (i < gates) {
    const int j = i - g0, q = f1_q(j, dr);
    return f1_code(1, 1 + q, j - q * tiles_r);
  }
  const int t = i - gates, q = f1_q(t, dn);
  return f1_code(0, q, t - q * ndn);
}

// Waits (bounded) until *cnt >= need; acquire.
__device__ __forceinline__ bool wait_count(const unsigned* cnt, unsigned need) {
  if (ld_acquire_gpu(cnt) >= need) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire_gpu(cnt) >= need) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

}  // namespace

}  // namespace moe
