// rvq.cu -- decode for layers whose experts are stored as 3-bit residual VQ.
//
// WASTE page, section "Quantization ve doğruluk": every run of 8 weights
// along a row is the sum of one codeword from each of 3 stages, each stage a
// codebook of 256 eight-value codewords, so a row carries 3 code bytes per 8
// weights (3.00 bits per weight).  The layer's codebooks (bf16, one set of 3
// stages for each of gate, up and down) stay resident next to the router;
// the records hold only code bytes:
//   [gate codes F x 3H/8][up codes F x 3H/8][down codes H x 3F/8]
// row-major, a row's blocks in order, each block's stage bytes in order.
//
// The page's method: the dot product of the input with every codeword is
// tabulated once per block of 8 inputs, and each row then costs three table
// lookups and their sum per block, with no weight rebuilt.  Here the input is
// cut into slices of 32 blocks (256 inputs); a CTA tabulates one slice,
//   T[stage][block][code] = <codeword(stage, code), x_block>,
// 96 KB per matrix kind in shared memory, and streams the code bytes of its
// share of the rows, one row per thread, adding one table entry per stage
// and block.  Partial sums per slice land in the workspace and small kernels
// add them in a fixed order.  Per token:
//   rvq_gateup_kernel   (slice, row part): gate and up partial sums of every
//                       active expert and the shared expert
//   rvq_swiglu_kernel   h = silu(sum g) * (sum u)
//   rvq_down_kernel     (expert entry, slice of F, row part): down partials
//   rvq_combine_kernel  out = sum_i p_i y_i + y_shared, bf16 and f32
// A lookup's index is the code byte, so the 32 lanes of a warp hit random
// banks: about 3.5 shared-memory wavefronts per lookup instruction, which
// bounds these kernels below the HBM rate.
#include <algorithm>
#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

cudaError_t launch_decode_router(const LayerArgs& a, int num_sms, cudaStream_t st);

namespace {

constexpr int kRvqThreads = 256;
constexpr int kTB = 32;          // blocks of 8 inputs per slice
constexpr int kCodes = 256;      // codewords per stage
constexpr int kKindWords = 3 * kCodes;
constexpr int kTabFloats = 3 * kTB * kCodes;  // one kind's table of a slice

// Launch geometry of one token, the same on host and device.
struct RvqPlan {
  int S, P, rpp;          // gate|up: input slices, row parts, rows per part
  int Sdr, Sds, Sdm, Pd;  // down: slices of F, of Fs, their maximum; row parts
  int rpd;                // down rows per part
};

int cdiv(int a, int b) { return (a + b - 1) / b; }

RvqPlan rvq_plan(const LayerArgs& a, int num_sms) {
  RvqPlan p;
  const int R = a.k * a.F + a.Fs;
  p.S = cdiv(a.H / 8, kTB);
  p.P = std::max(1, std::min(num_sms / p.S, cdiv(R, kRvqThreads)));  // one CTA per SM
  p.rpp = cdiv(R, p.P);
  p.Sdr = cdiv(a.F / 8, kTB);
  p.Sds = a.Fs ? cdiv(a.Fs / 8, kTB) : 0;
  p.Sdm = std::max(p.Sdr, p.Sds);
  p.Pd = std::max(1, std::min(2 * num_sms / (a.k * p.Sdr + p.Sds), cdiv(a.H, kRvqThreads)));  // two per SM
  p.rpd = cdiv(a.H, p.Pd);
  return p;
}

size_t gateup_smem() { return (2 * kTabFloats + kTB * 8) * sizeof(float); }
size_t down_smem() { return (kTabFloats + kTB * 8) * sizeof(float); }

__device__ __forceinline__ float rvq_silu(float g) { return g / (1.0f + expf(-g)); }

// T[kind][stage][j][c] = <codeword(kind, stage, c), v[8j .. 8j+7]> for
// nkinds kinds starting at book (bf16 codewords as uint4) and nb blocks.
__device__ __forceinline__ void build_tables(const uint4* __restrict__ book, int nkinds,
                                             const float* __restrict__ v, int nb, float* __restrict__ T) {
  for (int q = threadIdx.x; q < nkinds * kKindWords; q += kRvqThreads) {
    const int c = q % kCodes, ks = q / kCodes;  // ks = kind * 3 + stage
    const uint4 w = __ldg(book + q);
    const float c0 = bf16lo(w.x), c1 = bf16hi(w.x), c2 = bf16lo(w.y), c3 = bf16hi(w.y);
    const float c4 = bf16lo(w.z), c5 = bf16hi(w.z), c6 = bf16lo(w.w), c7 = bf16hi(w.w);
    float* out = T + static_cast<size_t>(ks) * kTB * kCodes + c;
    for (int j = 0; j < nb; ++j) {
      const float* x = v + 8 * j;
      float d = c0 * x[0];
      d = fmaf(c1, x[1], d), d = fmaf(c2, x[2], d), d = fmaf(c3, x[3], d);
      d = fmaf(c4, x[4], d), d = fmaf(c5, x[5], d), d = fmaf(c6, x[6], d), d = fmaf(c7, x[7], d);
      out[j * kCodes] = d;
    }
  }
}

// Sum over NB blocks and 3 stages of T[stage][j][code byte 3j + stage] for
// one row's 3*NB code bytes (8-byte aligned).
template <int NB>
__device__ __forceinline__ float lookup_row(const uint8_t* __restrict__ codes, const float* __restrict__ T) {
  constexpr int NW = 3 * NB / 8;
  uint2 w[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) w[i] = __ldg(reinterpret_cast<const uint2*>(codes) + i);
  float acc[3] = {0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < NB; ++j)
#pragma unroll
    for (int s = 0; s < 3; ++s) {
      const int n = 3 * j + s;
      const uint32_t word = (n % 8) < 4 ? w[n / 8].x : w[n / 8].y;
      acc[s] += T[(s * kTB + j) * kCodes + ((word >> (8 * (n % 4))) & 0xFFu)];
    }
  return (acc[0] + acc[1]) + acc[2];
}

// Rows [r0, r1) of the gate|up matrices of every entry (entry-major: routed
// entries' F rows in rank order, then the shared expert's Fs rows), over one
// slice of the input.
template <int NB>
__device__ void gateup_rows(const LayerArgs& a, int t, int slice, int r0, int r1, const float* T) {
  const int Fm = max(a.F, a.Fs);
  const size_t row_bytes = static_cast<size_t>(a.H) / 8 * 3, o0 = static_cast<size_t>(slice) * kTB * 3;
  for (int r = r0 + threadIdx.x; r < r1; r += kRvqThreads) {
    int e, f;
    const uint8_t* rec;
    const RecordOffsets* off;
    if (r < a.k * a.F) {
      e = r / a.F, f = r - e * a.F, off = &a.off_r;
      rec = a.records + static_cast<size_t>(a.ids[t * a.k + e]) * a.off_r.stride;
    } else {
      e = a.k, f = r - a.k * a.F, off = &a.off_s, rec = a.shared;
    }
    const size_t o = static_cast<size_t>(f) * row_bytes + o0;
    const float g = lookup_row<NB>(rec + off->gate_codes + o, T);
    const float u = lookup_row<NB>(rec + off->up_codes + o, T + kTabFloats);
    const size_t idx = (static_cast<size_t>(slice) * (a.k + 1) + e) * Fm + f;
    a.ws.rvq_g[idx] = g, a.ws.rvq_u[idx] = u;
  }
}

// grid S * P: CTA (slice, part)
__global__ void __launch_bounds__(kRvqThreads, 1) rvq_gateup_kernel(const __grid_constant__ LayerArgs a,
                                                                     const RvqPlan pl, int t) {
  extern __shared__ __align__(16) float smem[];
  float* T = smem;                   // [gate, up][3][kTB][256]
  float* xs = smem + 2 * kTabFloats;  // the slice's inputs
  const int slice = blockIdx.x % pl.S, part = blockIdx.x / pl.S;
  const int b0 = slice * kTB, nb = min(kTB, a.H / 8 - b0);
  const uint16_t* x = a.x + static_cast<size_t>(t) * a.H + 8 * b0;
  for (int i = threadIdx.x; i < nb * 8; i += kRvqThreads) xs[i] = __uint_as_float(static_cast<uint32_t>(x[i]) << 16);
  __syncthreads();
  build_tables(reinterpret_cast<const uint4*>(a.cbs), 2, xs, nb, T);
  __syncthreads();
  const int R = a.k * a.F + a.Fs, r0 = part * pl.rpp, r1 = min(R, r0 + pl.rpp);
  switch (nb) {  // a.H is a multiple of 64: whole slices, or a last one of 8, 16 or 24 blocks
    case 32: gateup_rows<32>(a, t, slice, r0, r1, T); break;
    case 24: gateup_rows<24>(a, t, slice, r0, r1, T); break;
    case 16: gateup_rows<16>(a, t, slice, r0, r1, T); break;
    default: gateup_rows<8>(a, t, slice, r0, r1, T); break;
  }
}

// grid ceil((k F + Fs) / 256): h of every entry from the slices' partial sums
__global__ void __launch_bounds__(kRvqThreads) rvq_swiglu_kernel(const __grid_constant__ LayerArgs a,
                                                                 const RvqPlan pl, int t) {
  const int r = blockIdx.x * kRvqThreads + threadIdx.x;
  if (r >= a.k * a.F + a.Fs) return;
  const int Fm = max(a.F, a.Fs);
  const int e = r < a.k * a.F ? r / a.F : a.k, f = r < a.k * a.F ? r - e * a.F : r - a.k * a.F;
  float g = 0.f, u = 0.f;
  for (int sl = 0; sl < pl.S; ++sl) {
    const size_t idx = (static_cast<size_t>(sl) * (a.k + 1) + e) * Fm + f;
    g += a.ws.rvq_g[idx], u += a.ws.rvq_u[idx];
  }
  const float h = rvq_silu(g) * u;
  if (e < a.k) a.ws.h[(static_cast<size_t>(t) * a.k + e) * a.F + f] = h;
  else a.ws.h_shared[static_cast<size_t>(t) * a.Fs + f] = h;
}

template <int NB>
__device__ void down_rows(const LayerArgs& a, const uint8_t* codes, size_t row_bytes, int r0, int r1,
                          float* y, const float* T) {
  for (int r = r0 + threadIdx.x; r < r1; r += kRvqThreads)
    y[r] = lookup_row<NB>(codes + static_cast<size_t>(r) * row_bytes, T);
}

// grid k * Sdr * Pd + Sds * Pd: CTA (entry, slice of the entry's F, row part)
__global__ void __launch_bounds__(kRvqThreads, 2) rvq_down_kernel(const __grid_constant__ LayerArgs a,
                                                                  const RvqPlan pl, int t) {
  extern __shared__ __align__(16) float smem[];
  float* T = smem;             // [3][kTB][256]
  float* hs = smem + kTabFloats;
  int e, slice, part, Fe;
  const uint8_t* rec;
  const RecordOffsets* off;
  const float* h;
  const int nr = a.k * pl.Sdr * pl.Pd;
  if (static_cast<int>(blockIdx.x) < nr) {
    const int per = pl.Sdr * pl.Pd, rem = blockIdx.x % per;
    e = blockIdx.x / per, slice = rem % pl.Sdr, part = rem / pl.Sdr, Fe = a.F, off = &a.off_r;
    rec = a.records + static_cast<size_t>(a.ids[t * a.k + e]) * a.off_r.stride;
    h = a.ws.h + (static_cast<size_t>(t) * a.k + e) * a.F;
  } else {
    const int i = blockIdx.x - nr;
    e = a.k, slice = i % pl.Sds, part = i / pl.Sds, Fe = a.Fs, off = &a.off_s, rec = a.shared;
    h = a.ws.h_shared + static_cast<size_t>(t) * a.Fs;
  }
  const int b0 = slice * kTB, nb = min(kTB, Fe / 8 - b0);
  for (int i = threadIdx.x; i < nb * 8; i += kRvqThreads) hs[i] = h[8 * b0 + i];
  __syncthreads();
  build_tables(reinterpret_cast<const uint4*>(a.cbs) + 2 * kKindWords, 1, hs, nb, T);
  __syncthreads();
  const size_t row_bytes = static_cast<size_t>(Fe) / 8 * 3;
  const uint8_t* codes = rec + off->down_codes + static_cast<size_t>(b0) * 3;
  float* y = a.ws.rvq_y + (static_cast<size_t>(e) * pl.Sdm + slice) * a.H;
  const int r0 = part * pl.rpd, r1 = min(a.H, r0 + pl.rpd);
  switch (nb) {
    case 32: down_rows<32>(a, codes, row_bytes, r0, r1, y, T); break;
    case 24: down_rows<24>(a, codes, row_bytes, r0, r1, y, T); break;
    case 16: down_rows<16>(a, codes, row_bytes, r0, r1, y, T); break;
    default: down_rows<8>(a, codes, row_bytes, r0, r1, y, T); break;
  }
}

// grid ceil(H / 256): out = sum_i p_i y_i + y_shared, entries in rank order
__global__ void __launch_bounds__(kRvqThreads) rvq_combine_kernel(const __grid_constant__ LayerArgs a,
                                                                  const RvqPlan pl, int t) {
  const int r = blockIdx.x * kRvqThreads + threadIdx.x;
  if (r >= a.H) return;
  float acc = 0.f;
  for (int i = 0; i < a.k; ++i) {
    float y = 0.f;
    for (int sl = 0; sl < pl.Sdr; ++sl) y += a.ws.rvq_y[(static_cast<size_t>(i) * pl.Sdm + sl) * a.H + r];
    acc = fmaf(a.weights[t * a.k + i], y, acc);
  }
  if (a.Fs) {
    float y = 0.f;
    for (int sl = 0; sl < pl.Sds; ++sl) y += a.ws.rvq_y[(static_cast<size_t>(a.k) * pl.Sdm + sl) * a.H + r];
    acc += y;
  }
  a.out_bf16[static_cast<size_t>(t) * a.H + r] = f32_to_bf16_rne(acc);
  if (a.out_f32) a.out_f32[static_cast<size_t>(t) * a.H + r] = acc;
}

}  // namespace

size_t rvq_smem_need(const LayerArgs&) { return std::max(gateup_smem(), down_smem()); }

cudaError_t set_rvq_attributes(int smem_optin) {
  cudaError_t e = cudaFuncSetAttribute(rvq_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
  return e ? e : cudaFuncSetAttribute(rvq_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
}

cudaError_t launch_decode_rvq(const LayerArgs& a, int num_sms, cudaStream_t st) {
  cudaError_t e = launch_decode_router(a, num_sms, st);
  if (e) return e;
  const RvqPlan pl = rvq_plan(a, num_sms);
  const int R = a.k * a.F + a.Fs;
  for (int t = 0; t < a.T; ++t) {
    rvq_gateup_kernel<<<pl.S * pl.P, kRvqThreads, gateup_smem(), st>>>(a, pl, t);
    rvq_swiglu_kernel<<<cdiv(R, kRvqThreads), kRvqThreads, 0, st>>>(a, pl, t);
    rvq_down_kernel<<<a.k * pl.Sdr * pl.Pd + pl.Sds * pl.Pd, kRvqThreads, down_smem(), st>>>(a, pl, t);
    rvq_combine_kernel<<<cdiv(a.H, kRvqThreads), kRvqThreads, 0, st>>>(a, pl, t);
    if ((e = cudaGetLastError())) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
