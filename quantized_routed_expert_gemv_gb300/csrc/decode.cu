// decode.cu -- CUDA-core kernels of the MoE FFN decode step (sm_103a).
//
//   router_kernel   8-bit affine router GEMV -> fp32 logits; the last CTA to
//                   finish runs softmax + warp-shuffle top-k per token and
//                   groups the (token, slot) pairs by expert.
//   gateup_kernel   4-bit gate|up GEMV + SwiGLU for every active expert and
//                   the shared expert; each expert's rows are read once per
//                   step and applied to all of its tokens.
//   down_kernel     4-bit down GEMV into per-(token, slot) partials; the last
//                   CTA to finish a row tile combines the tile in fixed slot
//                   order (weighted routed outputs + shared output).
//
// The method follows the TurboFieldfare page, section "Token üretim süreci"
// (router on resident weights, top-8 ids, shared expert, combine; one
// fetched expert serves several rows) and section "Belleği azaltan çalışma
// yapısı" (affine 4-bit group-64 experts, 8-bit router); the record holds
// gate, up and down contiguously as on the WASTE page, section "Disk
// streaming mimarisi".
//
// GEMV inner loop.  A code q in bits [4i, 4i+4) of a 32-bit word, isolated
// by one AND, reads as the fp32 value q * 2^(4i-149) (bit patterns below
// 2^24 are subnormal or the first binade, both exact multiples of 2^-149).
// Activations are pre-scaled once per column by 2^(85-4i) so every product
// is q*x*2^-64 and one packed FMA (fma.rn.f32x2) handles two codes; the
// factored affine term is y = sum_g (s_g 2^64 dot_g + b_g sum_g x).  No
// integer-to-float conversion and no per-code scale multiply remain.
// Nibbles 6 and 7 are shifted down by 8 bits first (positions 4 and 5).
#include <algorithm>
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// Pre-scale of the activation multiplying nibble i of a word (i = 0..7).
__device__ __forceinline__ constexpr float nib_scale(int i) {
  return i == 0 ? 0x1p85f
         : i == 1 ? 0x1p81f
         : i == 2 ? 0x1p77f
         : i == 3 ? 0x1p73f
         : (i == 4 || i == 6) ? 0x1p69f
                              : 0x1p65f;
}

// 32 4-bit codes (16 bytes) against 32 pre-scaled activations: returns
// sum q_m x_m * 2^-64.
__device__ __forceinline__ float dot32(const uint4 q, const float (&X)[32]) {
  float a0 = 0.f, a1 = 0.f;
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = w[i], u = v >> 8;
    ffma2(a0, a1, __uint_as_float(v & 0x0000000Fu), __uint_as_float(v & 0x000000F0u),
          X[8 * i + 0], X[8 * i + 1]);
    ffma2(a0, a1, __uint_as_float(v & 0x00000F00u), __uint_as_float(v & 0x0000F000u),
          X[8 * i + 2], X[8 * i + 3]);
    ffma2(a0, a1, __uint_as_float(v & 0x000F0000u), __uint_as_float(v & 0x00F00000u),
          X[8 * i + 4], X[8 * i + 5]);
    ffma2(a0, a1, __uint_as_float(u & 0x000F0000u), __uint_as_float(u & 0x00F00000u),
          X[8 * i + 6], X[8 * i + 7]);
  }
  return a0 + a1;
}

// 32 bf16 activations (64 bytes, 64-byte aligned) -> pre-scaled fp32 + sum.
__device__ __forceinline__ void load_x_bf16(const uint16_t* p, float (&X)[32], float& SX) {
  const uint4* v = reinterpret_cast<const uint4*>(p);
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 t = __ldg(v + i);
    w[4 * i + 0] = t.x, w[4 * i + 1] = t.y, w[4 * i + 2] = t.z, w[4 * i + 3] = t.w;
  }
  float s = 0.f;
#pragma unroll
  for (int m = 0; m < 32; ++m) {
    const float x = (m & 1) ? bf16hi(w[m >> 1]) : bf16lo(w[m >> 1]);
    X[m] = x * nib_scale(m & 7);
    s += x;
  }
  SX = s;
}

// 32 fp32 activations (128 bytes, written by an earlier kernel).
__device__ __forceinline__ void load_x_f32(const float* p, float (&X)[32], float& SX) {
  const float4* v = reinterpret_cast<const float4*>(p);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 t = __ldcg(v + i);
    const float e[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = 4 * i + j;
      X[m] = e[j] * nib_scale(m & 7);
      s += e[j];
    }
  }
  SX = s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// ============================================================================
// Router: logits, then (last CTA) top-k, weights and grouping by expert.
// ============================================================================

// 16 8-bit codes (16 bytes) against pre-scaled activations: byte i of a word
// isolated by one AND reads as q * 2^(8i-149) for i = 0..2; byte 3 is shifted
// down by 8 bits first.  Activation pre-scales 2^85, 2^77, 2^69, 2^69.
__device__ __forceinline__ constexpr float byte_scale(int i) {
  return i == 0 ? 0x1p85f : i == 1 ? 0x1p77f : 0x1p69f;
}

__device__ __forceinline__ float dot16_u8(const uint4 q, const float (&X)[16]) {
  float a0 = 0.f, a1 = 0.f;
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = w[i];
    ffma2(a0, a1, __uint_as_float(v & 0x000000FFu), __uint_as_float(v & 0x0000FF00u),
          X[4 * i + 0], X[4 * i + 1]);
    ffma2(a0, a1, __uint_as_float(v & 0x00FF0000u), __uint_as_float((v >> 8) & 0x00FF0000u),
          X[4 * i + 2], X[4 * i + 3]);
  }
  return a0 + a1;
}

template <int NT>
__global__ void __launch_bounds__(256) router_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(16) float rsm[];
  pdl_launch_dependents();
  const int H = a.H, E = a.E, T = a.T, k = a.k;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nchunk = H >> 4;  // 16-byte chunks per router row
  const int gw = blockIdx.x * 8 + warp, nw = gridDim.x * 8;

  for (int e = gw; e < E; e += nw) {
    const uint4* crow = reinterpret_cast<const uint4*>(a.rcodes + static_cast<size_t>(e) * H);
    const uint32_t* srow = a.rsb + static_cast<size_t>(e) * (H >> 6);
    for (int t0 = 0; t0 < T; t0 += NT) {
      float acc[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t] = 0.f;
      for (int c = lane; c < nchunk; c += 32) {
        const uint4 q = __ldg(crow + c);
        const uint32_t sbw = __ldg(srow + (c >> 2));
        const float s = bf16lo(sbw) * 0x1p64f, b = bf16hi(sbw);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t0 + t < T) {
            const uint4* xp =
                reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t0 + t) * H + c * 16);
            const uint4 x0 = __ldg(xp), x1 = __ldg(xp + 1);
            const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            float X[16], sx = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
              const float xv = (m & 1) ? bf16hi(xw[m >> 1]) : bf16lo(xw[m >> 1]);
              X[m] = xv * byte_scale(m & 3);
              sx += xv;
            }
            acc[t] = fmaf(s, dot16_u8(q, X), fmaf(b, sx, acc[t]));
          }
        }
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float v = warp_sum(acc[t]);
        if (lane == 0 && t0 + t < T)
          a.ws.logits[static_cast<size_t>(t0 + t) * E + e] = v + (a.beta ? __ldg(a.beta + e) : 0.f);
      }
    }
  }

  // ---- last CTA: top-k, weights, grouping --------------------------------
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&a.ws.ctl[1], 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  float* Lw = rsm + warp * E;                                     // per-warp logits
  unsigned* sel = reinterpret_cast<unsigned*>(rsm + 8 * E);       // [E][4] token bitmasks
  int* s_off = reinterpret_cast<int*>(sel + 4 * E);               // [E] pair offsets
  int* s_ids = s_off + E;                                         // [T*k]
  int* s_scan = s_ids + kMaxTokens * kMaxTopK;                    // [16] scan scratch

  for (int i = tid; i < 4 * E; i += 256) sel[i] = 0u;
  __syncthreads();

  for (int t = warp; t < T; t += 8) {
    for (int e = lane; e < E; e += 32) Lw[e] = __ldcg(a.ws.logits + static_cast<size_t>(t) * E + e);
    __syncwarp();
    float myl = 0.f;
    int myi = 0;
    for (int i = 0; i < k; ++i) {
      float bv = -FLT_MAX;
      int bi = E;
      for (int e = lane; e < E; e += 32) {
        const float v = Lw[e];
        if (v > bv || (v == bv && e < bi)) bv = v, bi = e;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) bv = ov, bi = oi;
      }
      if (bi >= E) {  // only reachable with non-finite logits (outside the contract)
        if (lane == 0) latch_error(&a.ws.ctl[0], kErrRange);
        bi = i;
      }
      if (lane == i) myl = bv, myi = bi;
      __syncwarp();
      if (lane == 0) Lw[bi] = -INFINITY;
      __syncwarp();
    }
    const float lmax = __shfl_sync(0xFFFFFFFFu, myl, 0);
    const float ex = (lane < k) ? expf(myl - lmax) : 0.f;
    const float z = warp_sum(ex);
    if (lane < k) {
      a.ids[t * k + lane] = myi;
      a.weights[t * k + lane] = ex / z;
      s_ids[t * k + lane] = myi;
      atomicOr(&sel[myi * 4 + (t >> 5)], 1u << (t & 31));
    }
    __syncwarp();
  }
  __syncthreads();

  // counts, exclusive scans over experts (pairs and active experts)
  const int ept = (E + 255) / 256;
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
    const int cu = __shfl_up_sync(0xFFFFFFFFu, c_inc, o);
    const int au = __shfl_up_sync(0xFFFFFFFFu, a_inc, o);
    if (lane >= o) c_inc += cu, a_inc += au;
  }
  if (lane == 31) s_scan[warp] = c_inc, s_scan[8 + warp] = a_inc;
  __syncthreads();
  int c_base = 0, a_base = 0;
  for (int w = 0; w < warp; ++w) c_base += s_scan[w], a_base += s_scan[8 + w];
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
  if (tid == 255) *a.ws.n_act = a_run;
  __syncthreads();

  for (int p = tid; p < T * k; p += 256) {
    const int t = p / k, e = s_ids[p];
    int rank = 0;
    for (int w = 0; w < (t >> 5); ++w) rank += __popc(sel[4 * e + w]);
    rank += __popc(sel[4 * e + (t >> 5)] & ((1u << (t & 31)) - 1u));
    const int pos = s_off[e] + rank;
    a.ws.pair_token[pos] = t;
    a.ws.pair_slot[pos] = p;
  }
  if (tid == 0) a.ws.ctl[1] = 0u;  // counter back to zero for the next call
}

// ============================================================================
// Shared machinery of the two expert GEMV kernels.
// ============================================================================

struct Entry {     // one expert's work this step
  const uint8_t* rec;
  const RecordOffsets* off;  // points into the __grid_constant__ kernel parameter
  int Fe;          // FFN width of this expert (F or Fs)
  int ntok;        // tokens routed to it
  int pair0;       // first pair (routed) -- h row of token 0
  int shared;      // 1 for the shared expert
};

__device__ __forceinline__ Entry get_entry(const LayerArgs& a, int idx, int n_act, int has_sh) {
  Entry en;
  if (has_sh && idx == 0) {
    en.rec = a.shared, en.off = &a.off_s, en.Fe = a.Fs, en.ntok = a.T, en.pair0 = 0,
    en.shared = 1;
    return en;
  }
  const int i = idx - has_sh;
  int e = a.ws.act_expert[i];
  int cnt = a.ws.act_cnt[i];
  if (e < 0 || e >= a.E) e = 0;
  if (cnt < 0 || cnt > a.T) cnt = 0;
  const int slot = a.slot_of ? a.slot_of[e] : e;
  en.rec = a.records + static_cast<size_t>(slot) * a.off_r.stride;
  en.off = &a.off_r, en.Fe = a.F, en.ntok = cnt, en.pair0 = a.ws.act_off[i], en.shared = 0;
  return en;
}

__device__ __forceinline__ int entry_token(const LayerArgs& a, const Entry& en, int t) {
  return en.shared ? t : a.ws.pair_token[en.pair0 + t];
}

// ============================================================================
// gate|up + SwiGLU.  One item = `rth` gate rows and the same `rth` up rows of
// one expert; the shared expert's items come first.
// ============================================================================

template <int NTOK>
__global__ void __launch_bounds__(kConsumers + 32, 1) gateup_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.H, C = H >> 5, NRL = kConsumers / C;
  const int max_rows = 2 * max(a.rth_r, a.rth_s);
  float* red = reinterpret_cast<float*>(smem + kStages * a.stage_bytes);  // [NTOK][rows][C]
  float* yv = red + NTOK * max_rows * C;                                  // [NTOK][rows]
  uint64_t* full = reinterpret_cast<uint64_t*>(yv + NTOK * max_rows);
  uint64_t* empty = full + kStages;
  volatile int* s_abort = reinterpret_cast<volatile int*>(empty + kStages);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1), mbar_init(&empty[s], kConsumers / 32);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();  // router outputs (active experts, pairs) are ready past this point

  const int has_sh = a.Fs > 0 ? 1 : 0;
  const int n_act = min(*reinterpret_cast<volatile int*>(a.ws.n_act), a.E);
  const int tiles_r = a.F / a.rth_r, tiles_s = has_sh ? a.Fs / a.rth_s : 0;
  const int n_items = tiles_s + n_act * tiles_r;

  auto item = [&](int i, int& idx, int& tile) {
    if (i < tiles_s) idx = 0, tile = i;
    else idx = has_sh + (i - tiles_s) / tiles_r, tile = (i - tiles_s) % tiles_r;
  };

  if (warp == kConsumers / 32) {  // ---------------- producer warp
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++it) {
        const int s = it % kStages;
        if (it >= kStages && !mbar_wait(&empty[s], ((it / kStages) - 1) & 1)) {
          latch_error(&a.ws.ctl[0], kErrTimeout);
          break;
        }
        int idx, tile;
        item(i, idx, tile);
        const Entry en = get_entry(a, idx, n_act, has_sh);
        if (!en.shared && a.slot_tag) {
          const int e = a.ws.act_expert[idx - has_sh];
          if (a.slot_tag[a.slot_of[e]] != e) latch_error(&a.ws.ctl[0], kErrResidency);
        }
        const int rth = en.shared ? a.rth_s : a.rth_r;
        const size_t j0 = static_cast<size_t>(tile) * rth;
        const uint32_t cb = rth * (H / 2), sbb = rth * (H / 16);
        uint8_t* st = smem + s * a.stage_bytes;
        mbar_arrive_expect_tx(&full[s], 2 * cb + 2 * sbb);
        bulk_g2s(st, en.rec + en.off->gate_codes + j0 * (H / 2), cb, &full[s], pol);
        bulk_g2s(st + cb, en.rec + en.off->up_codes + j0 * (H / 2), cb, &full[s], pol);
        bulk_g2s(st + 2 * cb, en.rec + en.off->gate_sb + j0 * (H / 16), sbb, &full[s], pol);
        bulk_g2s(st + 2 * cb + sbb, en.rec + en.off->up_sb + j0 * (H / 16), sbb, &full[s], pol);
      }
      // every issued copy must land before this CTA may exit
      for (int j = max(0, it - kStages); j < it; ++j)
        if (!mbar_wait(&full[j % kStages], (j / kStages) & 1)) latch_error(&a.ws.ctl[0], kErrTimeout);
    }
    return;
  }

  // ---------------------------------------------------- consumer warps
  const int col = tid % C, rl = tid / C;
  const bool active = rl < NRL;
  float X[NTOK][32], SX[NTOK];
  const bool single = (a.T == 1);  // every entry's only token is token 0
  if (single && active) {
    load_x_bf16(a.x + col * 32, X[0], SX[0]);
#pragma unroll
    for (int t = 1; t < NTOK; ++t) {
#pragma unroll
      for (int m = 0; m < 32; ++m) X[t][m] = 0.f;
      SX[t] = 0.f;
    }
  }

  int it = 0;
  for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++it) {
    const int s = it % kStages;
    if (!mbar_wait(&full[s], (it / kStages) & 1)) *s_abort = 1;
    named_bar(1, kConsumers);
    if (*s_abort) {
      if (tid == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
      break;
    }
    int idx, tile;
    item(i, idx, tile);
    const Entry en = get_entry(a, idx, n_act, has_sh);
    const int rth = en.shared ? a.rth_s : a.rth_r;
    const int rows = 2 * rth;
    const uint8_t* st = smem + s * a.stage_bytes;
    const uint8_t* stsb = st + rows * (H / 2);
    float* hout = en.shared ? a.ws.h_shared : a.ws.h;
    const int j0 = tile * rth;

    for (int tg = 0; tg < en.ntok; tg += NTOK) {
      if (!single && active) {
#pragma unroll
        for (int t = 0; t < NTOK; ++t) {
          if (tg + t < en.ntok) {
            const int tok = entry_token(a, en, tg + t);
            load_x_bf16(a.x + static_cast<size_t>(tok) * H + col * 32, X[t], SX[t]);
          } else {
#pragma unroll
            for (int m = 0; m < 32; ++m) X[t][m] = 0.f;
            SX[t] = 0.f;
          }
        }
      }
      if (active) {
        for (int r = rl; r < rows; r += NRL) {
          const uint4 q = *reinterpret_cast<const uint4*>(st + r * (H / 2) + col * 16);
          const uint32_t sbw = *reinterpret_cast<const uint32_t*>(stsb + r * (H / 16) + (col >> 1) * 4);
          const float sc = bf16lo(sbw) * 0x1p64f, bi = bf16hi(sbw);
#pragma unroll
          for (int t = 0; t < NTOK; ++t)
            red[(t * rows + r) * C + col] = fmaf(sc, dot32(q, X[t]), bi * SX[t]);
        }
      }
      if (tg + NTOK >= en.ntok) {  // last pass over this stage: hand it back
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      named_bar(1, kConsumers);
      for (int p = warp; p < NTOK * rows; p += kConsumers / 32) {
        float v = 0.f;
        for (int c = lane; c < C; c += 32) v += red[p * C + c];
        v = warp_sum(v);
        if (lane == 0) yv[p] = v;
      }
      named_bar(1, kConsumers);
      for (int q = tid; q < NTOK * rth; q += kConsumers) {
        const int t = q / rth, j = q % rth;
        if (tg + t < en.ntok) {
          const float g = yv[t * rows + j], u = yv[t * rows + rth + j];
          const int hrow = en.shared ? (tg + t) : (en.pair0 + tg + t);
          hout[static_cast<size_t>(hrow) * en.Fe + j0 + j] = silu_f(g) * u;
        }
      }
    }
    if (en.ntok == 0) {  // cannot happen for a listed expert; keep the ring consistent
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}

// ============================================================================
// down + combine.  One item = `rt_down` rows of H of one expert.  Outputs go
// to ypart[token][slot][row]; the CTA whose arrival completes a row tile
// combines it: out = sum_i p_i y_i + y_shared, in slot order.
// ============================================================================

template <int NTOK>
__global__ void __launch_bounds__(kConsumers + 32, 1) down_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.H, RT = a.rt_down;
  const int Cmax = max(a.F, a.Fs) >> 5;
  float* red = reinterpret_cast<float*>(smem + kStages * a.stage_bytes);  // [NTOK][RT][C]
  float* yv = red + NTOK * RT * Cmax;                                     // [NTOK][RT]
  uint64_t* full = reinterpret_cast<uint64_t*>(yv + NTOK * RT);
  uint64_t* empty = full + kStages;
  volatile int* s_flags = reinterpret_cast<volatile int*>(empty + kStages);  // [0] abort [1] last
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1), mbar_init(&empty[s], kConsumers / 32);
    s_flags[0] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();  // h of every expert is ready past this point

  const int has_sh = a.Fs > 0 ? 1 : 0;
  const int n_act = min(*reinterpret_cast<volatile int*>(a.ws.n_act), a.E);
  const int n_entries = n_act + has_sh;
  const int n_tiles = a.n_tiles_down;
  const int n_items = n_entries * n_tiles;
  const int k = a.k;

  if (warp == kConsumers / 32) {  // ---------------- producer warp
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++it) {
        const int s = it % kStages;
        if (it >= kStages && !mbar_wait(&empty[s], ((it / kStages) - 1) & 1)) {
          latch_error(&a.ws.ctl[0], kErrTimeout);
          break;
        }
        const int idx = i / n_tiles, tile = i % n_tiles;
        const Entry en = get_entry(a, idx, n_act, has_sh);
        const size_t r0 = static_cast<size_t>(tile) * RT;
        const uint32_t cb = RT * (en.Fe / 2), sbb = RT * (en.Fe / 16);
        uint8_t* st = smem + s * a.stage_bytes;
        mbar_arrive_expect_tx(&full[s], cb + sbb);
        bulk_g2s(st, en.rec + en.off->down_codes + r0 * (en.Fe / 2), cb, &full[s], pol);
        bulk_g2s(st + cb, en.rec + en.off->down_sb + r0 * (en.Fe / 16), sbb, &full[s], pol);
      }
      for (int j = max(0, it - kStages); j < it; ++j)
        if (!mbar_wait(&full[j % kStages], (j / kStages) & 1)) latch_error(&a.ws.ctl[0], kErrTimeout);
    }
    return;
  }

  // ---------------------------------------------------- consumer warps
  float X[NTOK][32], SX[NTOK];
  int it = 0;
  for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++it) {
    const int s = it % kStages;
    if (!mbar_wait(&full[s], (it / kStages) & 1)) s_flags[0] = 1;
    named_bar(1, kConsumers);
    if (s_flags[0]) {
      if (tid == 0) latch_error(&a.ws.ctl[0], kErrTimeout);
      break;
    }
    const int idx = i / n_tiles, tile = i % n_tiles;
    const Entry en = get_entry(a, idx, n_act, has_sh);
    const int C = en.Fe >> 5, NRL = kConsumers / C;
    const int col = tid % C, rl = tid / C;
    const bool active = rl < NRL;
    const uint8_t* st = smem + s * a.stage_bytes;
    const uint8_t* stsb = st + RT * (en.Fe / 2);
    const float* hin = en.shared ? a.ws.h_shared : a.ws.h;
    const int r0 = tile * RT;

    for (int tg = 0; tg < en.ntok; tg += NTOK) {
      if (active) {
#pragma unroll
        for (int t = 0; t < NTOK; ++t) {
          if (tg + t < en.ntok) {
            const int hrow = en.shared ? (tg + t) : (en.pair0 + tg + t);
            load_x_f32(hin + static_cast<size_t>(hrow) * en.Fe + col * 32, X[t], SX[t]);
          } else {
#pragma unroll
            for (int m = 0; m < 32; ++m) X[t][m] = 0.f;
            SX[t] = 0.f;
          }
        }
        for (int r = rl; r < RT; r += NRL) {
          const uint4 q = *reinterpret_cast<const uint4*>(st + r * (en.Fe / 2) + col * 16);
          const uint32_t sbw =
              *reinterpret_cast<const uint32_t*>(stsb + r * (en.Fe / 16) + (col >> 1) * 4);
          const float sc = bf16lo(sbw) * 0x1p64f, bi = bf16hi(sbw);
#pragma unroll
          for (int t = 0; t < NTOK; ++t) red[(t * RT + r) * C + col] = fmaf(sc, dot32(q, X[t]), bi * SX[t]);
        }
      }
      if (tg + NTOK >= en.ntok) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      named_bar(1, kConsumers);
      for (int p = warp; p < NTOK * RT; p += kConsumers / 32) {
        float v = 0.f;
        for (int c = lane; c < C; c += 32) v += red[p * C + c];
        v = warp_sum(v);
        if (lane == 0) yv[p] = v;
      }
      named_bar(1, kConsumers);
      for (int q = tid; q < NTOK * RT; q += kConsumers) {
        const int t = q / RT, r = q % RT;
        if (tg + t < en.ntok) {
          int tok, slot;
          if (en.shared) {
            tok = tg + t, slot = k;
          } else {
            const int p = a.ws.pair_slot[en.pair0 + tg + t];
            tok = p / k, slot = p % k;
          }
          a.ws.ypart[(static_cast<size_t>(tok) * (k + 1) + slot) * H + r0 + r] = yv[q];
        }
      }
    }
    if (en.ntok == 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- arrival on the row tile; the last arriving CTA combines it
    __threadfence();
    named_bar(1, kConsumers);
    if (tid == 0) s_flags[1] = (atomicAdd(&a.ws.tile_cnt[tile], 1u) == static_cast<unsigned>(n_entries - 1));
    named_bar(1, kConsumers);
    if (s_flags[1]) {
      __threadfence();
      for (int q = tid; q < a.T * RT; q += kConsumers) {
        const int t = q / RT, r = r0 + q % RT;
        const float* yp = a.ws.ypart + static_cast<size_t>(t) * (k + 1) * H + r;
        float acc = 0.f;
        for (int i2 = 0; i2 < k; ++i2) acc = fmaf(__ldcg(a.weights + t * k + i2), __ldcg(yp + static_cast<size_t>(i2) * H), acc);
        if (has_sh) acc += __ldcg(yp + static_cast<size_t>(k) * H);
        a.out_bf16[static_cast<size_t>(t) * H + r] = f32_to_bf16_rne(acc);
        if (a.out_f32) a.out_f32[static_cast<size_t>(t) * H + r] = acc;
      }
      if (tid == 0) a.ws.tile_cnt[tile] = 0u;
    }
  }
}

// ============================================================================
// Host-side launchers (called from api.cu).
// ============================================================================

size_t router_smem_bytes(int E) {
  return static_cast<size_t>(8 * E) * 4 + static_cast<size_t>(4 * E) * 4 +
         static_cast<size_t>(E) * 4 + static_cast<size_t>(kMaxTokens * kMaxTopK) * 4 + 16 * 4;
}

size_t gateup_smem_bytes(const LayerArgs& a, int ntok) {
  const int max_rows = 2 * std::max(a.rth_r, a.rth_s);
  return static_cast<size_t>(kStages) * a.stage_bytes +
         static_cast<size_t>(ntok) * max_rows * (a.H / 32) * 4 + static_cast<size_t>(ntok) * max_rows * 4 +
         2 * kStages * 8 + 16;
}

size_t down_smem_bytes(const LayerArgs& a, int ntok) {
  const int cmax = std::max(a.F, a.Fs) / 32;
  return static_cast<size_t>(kStages) * a.stage_bytes +
         static_cast<size_t>(ntok) * a.rt_down * cmax * 4 + static_cast<size_t>(ntok) * a.rt_down * 4 +
         2 * kStages * 8 + 16;
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
  const void* fns[] = {(const void*)router_kernel<1>, (const void*)router_kernel<4>,
                       (const void*)gateup_kernel<1>, (const void*)gateup_kernel<4>,
                       (const void*)down_kernel<1>,   (const void*)down_kernel<4>};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
    if (e) return e;
  }
  return cudaSuccess;
}

static cudaError_t mark(const LayerArgs& a, int i, cudaStream_t st) {
  return a.prof_on ? cudaEventRecord(static_cast<cudaEvent_t>(a.prof[i]), st) : cudaSuccess;
}

cudaError_t launch_decode(const LayerArgs& a, int num_sms, cudaStream_t st) {
  const bool one = (a.T == 1);
  const bool pdl = !a.prof_on;
  const int rgrid = std::max(1, std::min((a.E + 7) / 8, 2 * num_sms));
  cudaError_t e;
  if ((e = mark(a, 0, st))) return e;
  e = launch_ex(one ? (const void*)router_kernel<1> : (const void*)router_kernel<4>, dim3(rgrid),
                dim3(256), router_smem_bytes(a.E), st, false, a);
  if (e || (e = mark(a, 1, st))) return e;
  e = launch_ex(one ? (const void*)gateup_kernel<1> : (const void*)gateup_kernel<4>, dim3(num_sms),
                dim3(kConsumers + 32), gateup_smem_bytes(a, one ? 1 : 4), st, pdl, a);
  if (e || (e = mark(a, 2, st))) return e;
  e = launch_ex(one ? (const void*)down_kernel<1> : (const void*)down_kernel<4>, dim3(num_sms),
                dim3(kConsumers + 32), down_smem_bytes(a, one ? 1 : 4), st, pdl, a);
  if (e) return e;
  return mark(a, 3, st);
}

}  // namespace moe
