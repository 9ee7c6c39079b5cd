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
// The page computes partial dot-product tables of the input against every
// codeword and then spends three table lookups per block.  On this GPU a
// lookup with a data-dependent index into shared memory costs a bank
// conflict in most warps, so these kernels instead rebuild each block's 8
// weights from three 16-byte codeword loads (codebooks in shared memory)
// and take the dot product in fp32 registers.
//
// Per call: the 8-bit router (decode.cu), then
//   rvq_gateup_kernel  one CTA per (token, expert entry, 32 rows of F):
//                      h = silu(W_g x) * (W_u x) into the workspace;
//   rvq_down_kernel    one CTA per (token, 32 rows of H): every entry's h in
//                      shared memory, y rows, and the combine
//                      out = sum_i p_i y_i + y_shared in a fixed order.
#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

cudaError_t launch_decode_router(const LayerArgs& a, int num_sms, cudaStream_t st);

namespace {

constexpr int kRvqWarps = 8;
constexpr int kRvqThreads = kRvqWarps * 32;
constexpr int kRvqRows = 32;                       // rows per CTA, both kernels
constexpr int kRvqRowsPerWarp = kRvqRows / kRvqWarps;
constexpr int kBookWords = 3 * 256;                // one kind's codewords (uint4 each)

__device__ __forceinline__ float rvq_silu(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ float rvq_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Byte n (0..11) of three little-endian words.
__device__ __forceinline__ uint32_t code_byte(const uint32_t (&w)[3], int n) {
  return (w[n >> 2] >> (8 * (n & 3))) & 0xFFu;
}

// Adds the 8 values of one bf16 codeword to acc.
__device__ __forceinline__ void add_codeword(const uint4& c, float (&acc)[8]) {
  acc[0] += bf16lo(c.x), acc[1] += bf16hi(c.x), acc[2] += bf16lo(c.y), acc[3] += bf16hi(c.y);
  acc[4] += bf16lo(c.z), acc[5] += bf16hi(c.z), acc[6] += bf16lo(c.w), acc[7] += bf16hi(c.w);
}

// Partial dot product of one lane over a row of an RVQ matrix with `cols`
// inputs: the lane takes 4 consecutive blocks (12 code bytes, three aligned
// words) per pass, the warp 128 blocks.  book: one kind's codebooks
// [3][256] uint4 in shared memory; v: the input vector in shared memory.
__device__ __forceinline__ float rvq_row_part(const uint8_t* __restrict__ row, int cols,
                                              const uint4* __restrict__ book,
                                              const float* __restrict__ v, int lane) {
  const int nblk = cols / 8;
  float acc = 0.0f;
  for (int b0 = lane * 4; b0 < nblk; b0 += 128) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(row + static_cast<size_t>(b0) * 3);
    const uint32_t w[3] = {__ldg(p), __ldg(p + 1), __ldg(p + 2)};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float wv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < 3; ++s) add_codeword(book[s * 256 + code_byte(w, 3 * q + s)], wv);
      const float4 x0 = *reinterpret_cast<const float4*>(v + (b0 + q) * 8);
      const float4 x1 = *reinterpret_cast<const float4*>(v + (b0 + q) * 8 + 4);
      acc = fmaf(wv[0], x0.x, acc), acc = fmaf(wv[1], x0.y, acc);
      acc = fmaf(wv[2], x0.z, acc), acc = fmaf(wv[3], x0.w, acc);
      acc = fmaf(wv[4], x1.x, acc), acc = fmaf(wv[5], x1.y, acc);
      acc = fmaf(wv[6], x1.z, acc), acc = fmaf(wv[7], x1.w, acc);
    }
  }
  return acc;
}

size_t gateup_smem(const LayerArgs& a) { return static_cast<size_t>(a.H) * 4 + 2 * kBookWords * 16; }

size_t down_smem(const LayerArgs& a) {
  return static_cast<size_t>(a.k * a.F + a.Fs) * 4 + kBookWords * 16;
}

// grid (k * F/32 + Fs/32, T)
__global__ void __launch_bounds__(kRvqThreads) rvq_gateup_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* xs = reinterpret_cast<float*>(smem);
  uint4* books = reinterpret_cast<uint4*>(smem + static_cast<size_t>(a.H) * 4);  // gate, up
  const int t = blockIdx.y, H = a.H;
  const int tiles_r = a.F / kRvqRows;
  int entry, tile, Fe;
  const uint8_t* rec;
  const RecordOffsets* off;
  if (static_cast<int>(blockIdx.x) < a.k * tiles_r) {
    entry = blockIdx.x / tiles_r, tile = blockIdx.x % tiles_r, Fe = a.F, off = &a.off_r;
    rec = a.records + static_cast<size_t>(a.ids[t * a.k + entry]) * a.off_r.stride;
  } else {
    entry = a.k, tile = blockIdx.x - a.k * tiles_r, Fe = a.Fs, off = &a.off_s;
    rec = a.shared;
  }
  for (int j = threadIdx.x; j < H; j += kRvqThreads) {
    const uint16_t b = a.x[static_cast<size_t>(t) * H + j];
    xs[j] = __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  const uint4* src = reinterpret_cast<const uint4*>(a.cbs);
  for (int i = threadIdx.x; i < 2 * kBookWords; i += kRvqThreads) books[i] = src[i];
  __syncthreads();

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const size_t row_bytes = static_cast<size_t>(H) / 8 * 3;
  float* hout = entry < a.k ? a.ws.h + (static_cast<size_t>(t) * a.k + entry) * a.F
                            : a.ws.h_shared + static_cast<size_t>(t) * a.Fs;
  for (int rr = 0; rr < kRvqRowsPerWarp; ++rr) {
    const int r = tile * kRvqRows + warp * kRvqRowsPerWarp + rr;
    if (r >= Fe) break;
    const float g = rvq_sum(rvq_row_part(rec + off->gate_codes + r * row_bytes, H, books, xs, lane));
    const float u = rvq_sum(rvq_row_part(rec + off->up_codes + r * row_bytes, H, books + kBookWords, xs, lane));
    if (lane == 0) hout[r] = rvq_silu(g) * u;
  }
}

// grid (H/32, T)
__global__ void __launch_bounds__(kRvqThreads) rvq_down_kernel(const __grid_constant__ LayerArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int t = blockIdx.y, H = a.H, k = a.k, F = a.F, Fs = a.Fs;
  float* hs = reinterpret_cast<float*>(smem);  // [k][F] then [Fs]
  uint4* book = reinterpret_cast<uint4*>(smem + static_cast<size_t>(k * F + Fs) * 4);
  const float* hr = a.ws.h + static_cast<size_t>(t) * k * F;
  for (int j = threadIdx.x; j < k * F; j += kRvqThreads) hs[j] = hr[j];
  for (int j = threadIdx.x; j < Fs; j += kRvqThreads) hs[k * F + j] = a.ws.h_shared[static_cast<size_t>(t) * Fs + j];
  const uint4* src = reinterpret_cast<const uint4*>(a.cbs) + 2 * kBookWords;
  for (int i = threadIdx.x; i < kBookWords; i += kRvqThreads) book[i] = src[i];
  __syncthreads();

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int rr = 0; rr < kRvqRowsPerWarp; ++rr) {
    const int r = blockIdx.x * kRvqRows + warp * kRvqRowsPerWarp + rr;
    if (r >= H) break;
    float acc = 0.0f;
    for (int i = 0; i < k; ++i) {
      const uint8_t* rec = a.records + static_cast<size_t>(a.ids[t * k + i]) * a.off_r.stride;
      const float y = rvq_sum(rvq_row_part(rec + a.off_r.down_codes + static_cast<size_t>(r) * (F / 8 * 3), F,
                                           book, hs + static_cast<size_t>(i) * F, lane));
      acc = fmaf(a.weights[t * k + i], y, acc);
    }
    if (Fs)
      acc += rvq_sum(rvq_row_part(a.shared + a.off_s.down_codes + static_cast<size_t>(r) * (Fs / 8 * 3), Fs,
                                  book, hs + static_cast<size_t>(k) * F, lane));
    if (lane == 0) {
      a.out_bf16[static_cast<size_t>(t) * H + r] = f32_to_bf16_rne(acc);
      if (a.out_f32) a.out_f32[static_cast<size_t>(t) * H + r] = acc;
    }
  }
}

}  // namespace

size_t rvq_smem_need(const LayerArgs& a) { return gateup_smem(a) > down_smem(a) ? gateup_smem(a) : down_smem(a); }

cudaError_t set_rvq_attributes(int smem_optin) {
  cudaError_t e = cudaFuncSetAttribute(rvq_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
  return e ? e : cudaFuncSetAttribute(rvq_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
}

cudaError_t launch_decode_rvq(const LayerArgs& a, int num_sms, cudaStream_t st) {
  cudaError_t e = launch_decode_router(a, num_sms, st);
  if (e) return e;
  const dim3 g1(a.k * (a.F / kRvqRows) + a.Fs / kRvqRows, a.T);
  rvq_gateup_kernel<<<g1, kRvqThreads, gateup_smem(a), st>>>(a);
  if ((e = cudaGetLastError())) return e;
  const dim3 g2(a.H / kRvqRows, a.T);
  rvq_down_kernel<<<g2, kRvqThreads, down_smem(a), st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
