// gemv.cuh -- inner loops of the quantised GEMV kernels (sm_103a).
//
// Float path (any token count): a code q in bits [4i, 4i+4) of a 32-bit
// word, isolated by one AND, reads as the fp32 value q * 2^(4i-149) (bit
// patterns below 2^24 are subnormal or the first binade, exact multiples of
// 2^-149).  Activations are pre-scaled once per column by 2^(85-4i) so each
// product is q*x*2^-64; nibbles 6 and 7 are shifted down by 8 bits first.
// The affine term is factored as y = sum_g (s_g 2^64 dot_g + b_g sum_g x).
//
// Fixed-point path (one token): a chunk of 32 activations is written as
// 16-bit fixed point X_j = rint(x_j / 2^e) with one power-of-two exponent e
// per chunk (|X_j| < 2^15), split into a signed high byte and an unsigned
// low byte (X = 256*hi + lo).  Codes widen to bytes with one AND per four
// (even nibbles: w & 0x0F0F0F0F, odd: (w >> 4) & 0x0F0F0F0F) and dp4a
// (u8 x s8, u8 x u8) accumulates sum_j q_j X_j exactly in int32; the sum is
// below 2^24 so its fp32 value is exact.  The result is scaled by s * 2^e.
// A bf16 activation is represented exactly unless it is more than 2^7 below
// its chunk's largest magnitude; the rounding then stays below 2^-15 of
// that magnitude.
//
// Grouped variant (the single-token down's h rows): each 8-value group, i.e.
// word i of every kind below, carries its own exponent, so the producer of
// the group needs no other group's values.  The dot keeps four exact integer
// sums, one per group, each scaled by its own 2^e.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace moe {

constexpr unsigned kFull = 0xFFFFFFFFu;

// Pre-scale of the activation multiplying nibble i of a word (i = 0..7).
__device__ __forceinline__ constexpr float nib_scale(int i) {
  return i == 0 ? 0x1p85f
         : i == 1 ? 0x1p81f
         : i == 2 ? 0x1p77f
         : i == 3 ? 0x1p73f
         : (i == 4 || i == 6) ? 0x1p69f
                              : 0x1p65f;
}

// 32 4-bit codes (16 bytes) against 32 pre-scaled activations held as 16
// float pairs (X[j] = activations 2j, 2j+1): returns sum q_m x_m * 2^-64 as
// four independent scalar-FMA chains (faster than packed FMA on this part).
__device__ __forceinline__ float dot32(const uint4 q, const float2 (&X)[16]) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = w[i], u = v >> 8;
    float& d0 = (i & 1) ? a2 : a0;
    float& d1 = (i & 1) ? a3 : a1;
    d0 = fmaf(__uint_as_float(v & 0x0000000Fu), X[4 * i + 0].x, d0);
    d1 = fmaf(__uint_as_float(v & 0x000000F0u), X[4 * i + 0].y, d1);
    d0 = fmaf(__uint_as_float(v & 0x00000F00u), X[4 * i + 1].x, d0);
    d1 = fmaf(__uint_as_float(v & 0x0000F000u), X[4 * i + 1].y, d1);
    d0 = fmaf(__uint_as_float(v & 0x000F0000u), X[4 * i + 2].x, d0);
    d1 = fmaf(__uint_as_float(v & 0x00F00000u), X[4 * i + 2].y, d1);
    d0 = fmaf(__uint_as_float(u & 0x000F0000u), X[4 * i + 3].x, d0);
    d1 = fmaf(__uint_as_float(u & 0x00F00000u), X[4 * i + 3].y, d1);
  }
  return (a0 + a1) + (a2 + a3);
}

__device__ __forceinline__ void zero_x(float2 (&X)[16], float& SX) {
#pragma unroll
  for (int j = 0; j < 16; ++j) X[j] = make_float2(0.f, 0.f);
  SX = 0.f;
}

// 32 bf16 activations (64 bytes) -> pre-scaled fp32 pairs + their plain sum.
__device__ __forceinline__ void load_x_bf16(const uint16_t* p, float2 (&X)[16], float& SX) {
  const uint4* v = reinterpret_cast<const uint4*>(p);
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 t = __ldg(v + i);
    w[4 * i + 0] = t.x, w[4 * i + 1] = t.y, w[4 * i + 2] = t.z, w[4 * i + 3] = t.w;
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {  // word j holds activations 2j (low half) and 2j+1
    const float x0 = bf16lo(w[j]), x1 = bf16hi(w[j]);
    X[j] = make_float2(x0 * nib_scale((2 * j) & 7), x1 * nib_scale((2 * j + 1) & 7));
    s += x0;
    s += x1;
  }
  SX = s;
}

// Activations of column `col` from a shared-memory h row stored chunk-
// interleaved: float4 number i (activations 4i..4i+3) of column c sits at
// float4 index i*C + c, so a warp's 32 lanes read 32 consecutive float4s.
__device__ __forceinline__ void load_h_smem(const float* row, int C, int col, float2 (&X)[16],
                                            float& SX) {
  const float4* v = reinterpret_cast<const float4*>(row);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 t = v[i * C + col];
    X[2 * i] = make_float2(t.x * nib_scale((4 * i) & 7), t.y * nib_scale((4 * i + 1) & 7));
    X[2 * i + 1] = make_float2(t.z * nib_scale((4 * i + 2) & 7), t.w * nib_scale((4 * i + 3) & 7));
    s += t.x;
    s += t.y;
    s += t.z;
    s += t.w;
  }
  SX = s;
}

// Index of element f in an h row of width Fe stored chunk-interleaved.
__device__ __forceinline__ int h_index(int f, int Fe) {
  const int col = f >> 5, m = f & 31;
  return (((m >> 2) * (Fe >> 5) + col) << 2) + (m & 3);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Sums four per-lane row partials over the warp.  On return lane L holds the
// warp total of row ((L >> 4) & 1) * 2 + ((L >> 3) & 1).
__device__ __forceinline__ float bfly4(float p0, float p1, float p2, float p3, int lane) {
  const bool hi16 = lane & 16;
  float k0 = hi16 ? p2 : p0, k1 = hi16 ? p3 : p1;
  const float s0 = hi16 ? p0 : p2, s1 = hi16 ? p1 : p3;
  k0 += __shfl_xor_sync(kFull, s0, 16);
  k1 += __shfl_xor_sync(kFull, s1, 16);
  const bool hi8 = lane & 8;
  float k = hi8 ? k1 : k0;
  const float s = hi8 ? k0 : k1;
  k += __shfl_xor_sync(kFull, s, 8);
  k += __shfl_xor_sync(kFull, k, 4);
  k += __shfl_xor_sync(kFull, k, 2);
  k += __shfl_xor_sync(kFull, k, 1);
  return k;
}


// 16 8-bit codes (16 bytes) against pre-scaled activations: byte i of a word
// isolated by one AND reads as q * 2^(8i-149) for i = 0..2; byte 3 is shifted
// down by 8 bits first.  Activation pre-scales 2^85, 2^77, 2^69, 2^69.
__device__ __forceinline__ constexpr float byte_scale(int i) {
  return i == 0 ? 0x1p85f : i == 1 ? 0x1p77f : 0x1p69f;
}

__device__ __forceinline__ float dot16_u8(const uint4 q, const float2 (&X)[8]) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = w[i];
    float& d0 = (i & 1) ? a2 : a0;
    float& d1 = (i & 1) ? a3 : a1;
    d0 = fmaf(__uint_as_float(v & 0x000000FFu), X[2 * i].x, d0);
    d1 = fmaf(__uint_as_float(v & 0x0000FF00u), X[2 * i].y, d1);
    d0 = fmaf(__uint_as_float(v & 0x00FF0000u), X[2 * i + 1].x, d0);
    d1 = fmaf(__uint_as_float((v >> 8) & 0x00FF0000u), X[2 * i + 1].y, d1);
  }
  return (a0 + a1) + (a2 + a3);
}


__device__ __forceinline__ int dp4a_us(uint32_t a_u8, uint32_t b_s8, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a_u8), "r"(b_s8), "r"(c));
  return d;
}

__device__ __forceinline__ int dp4a_uu(uint32_t a_u8, uint32_t b_u8, int c) {
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a_u8), "r"(b_u8), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack4(int b0, int b1, int b2, int b3) {
  return (static_cast<uint32_t>(b0) & 0xFFu) | ((static_cast<uint32_t>(b1) & 0xFFu) << 8) |
         ((static_cast<uint32_t>(b2) & 0xFFu) << 16) | (static_cast<uint32_t>(b3) << 24);
}

// Fixed-point form of the 32 activations of one 4-bit chunk (codes 32c..32c+31).
// Word i of the chunk holds codes 8i..8i+7; its even nibbles widen to the
// bytes of (w & 0x0F0F0F0F) and its odd nibbles to those of (w >> 4) & ....
struct XChunk {
  uint32_t eh[4], el[4], oh[4], ol[4];  // high/low bytes of even/odd activations
};

// 2^e such that max|x| / 2^e < 2^15 (1 for an all-zero row).
__device__ __forceinline__ float fixed_scale(float amax) {
  if (!(amax > 0.f)) return 1.f;
  int ex;
  frexpf(amax, &ex);  // amax = m * 2^ex, m in [0.5, 1)
  return ldexpf(1.f, ex - 15);
}

__device__ __forceinline__ int to_fixed(float x, float inv_scale) {
  const float v = rintf(x * inv_scale);
  return static_cast<int>(fminf(fmaxf(v, -32767.f), 32767.f));
}

__device__ __forceinline__ void make_xchunk(const float (&x)[32], float inv_scale, XChunk& X) {
  int q[32];
#pragma unroll
  for (int m = 0; m < 32; ++m) q[m] = to_fixed(x[m], inv_scale);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int* p = q + 8 * i;
    X.eh[i] = pack4(p[0] >> 8, p[2] >> 8, p[4] >> 8, p[6] >> 8);
    X.el[i] = pack4(p[0], p[2], p[4], p[6]);
    X.oh[i] = pack4(p[1] >> 8, p[3] >> 8, p[5] >> 8, p[7] >> 8);
    X.ol[i] = pack4(p[1], p[3], p[5], p[7]);
  }
}

// Exact sum_m q_m X_m over one 16-byte chunk of codes.
__device__ __forceinline__ int dot_chunk(const uint4 q, const XChunk& X) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  int ah = 0, al = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t ev = w[i] & 0x0F0F0F0Fu, od = (w[i] >> 4) & 0x0F0F0F0Fu;
    ah = dp4a_us(ev, X.eh[i], ah);
    al = dp4a_uu(ev, X.el[i], al);
    ah = dp4a_us(od, X.oh[i], ah);
    al = dp4a_uu(od, X.ol[i], al);
  }
  return ah * 256 + al;
}


// sum_i sc[i] * (exact sum over group i of q_m X_m): the grouped form.
__device__ __forceinline__ float dot_chunk_g(const uint4 q, const XChunk& X, const float (&sc)[4]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float r = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t ev = w[i] & 0x0F0F0F0Fu, od = (w[i] >> 4) & 0x0F0F0F0Fu;
    int ah = dp4a_us(ev, X.eh[i], 0), al = dp4a_uu(ev, X.el[i], 0);
    ah = dp4a_us(od, X.oh[i], ah);
    al = dp4a_uu(od, X.ol[i], al);
    r = fmaf(sc[i], static_cast<float>(ah * 256 + al), r);
  }
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Fixed-point chunk from 32 activations with its own exponent; returns 2^e.
__device__ __forceinline__ float make_xchunk_own(const float (&x)[32], XChunk& X) {
  float amax = 0.f;
#pragma unroll
  for (int m = 0; m < 32; ++m) amax = fmaxf(amax, fabsf(x[m]));
  const float scale = fixed_scale(amax);
  make_xchunk(x, 1.f / scale, X);
  return scale;
}

}  // namespace moe
