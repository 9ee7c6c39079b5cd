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
// cut into slices of 32 blocks (256 inputs) and a CTA tabulates one slice of
// one matrix kind, 96 KB of shared memory laid out [stage][code][block]:
// the 32 blocks of one (stage, code) fill one 128-byte row of the 32 banks.
// Lane j of a warp owns block j of the slice for every row, so its lookups
// always hit bank j and a warp's 32 lookups are one conflict-free wavefront
// whatever the codes are (with lanes owning rows instead, the code decides
// the bank and a lookup costs about 3.15 wavefronts).  Each lane reads its
// block's 3 code bytes of a row straight from global memory; a warp takes 8
// rows at a time and sums each row over its lanes with one 8-row butterfly.
// Partial sums per slice land in the workspace; later kernels add them in a
// fixed order.  One launch of each kernel serves every token of the step:
//   rvq_gateup_kernel   (token, kind, slice, row part): gate or up partial
//                       sums of the token's routed experts and the shared
//                       expert; the table is built before the wait for the
//                       router, so it overlaps the router
//   rvq_down_kernel     (token, entry, slice of F, row part): h of the slice
//                       from the gate|up partials (SwiGLU), its table, then
//                       down partial sums
//   rvq_combine_kernel  out = sum_i p_i y_i + y_shared, bf16 and f32
#include <algorithm>
#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

cudaError_t launch_decode_router(const LayerArgs& a, int num_sms, cudaStream_t st);

namespace {

constexpr int kRvqThreads = 512;          // 16 warps
constexpr int kRvqWarps = kRvqThreads / 32;
constexpr int kTB = 32;                   // blocks of 8 inputs per slice: one per lane
constexpr int kCodes = 256;               // codewords per stage
constexpr int kKindWords = 3 * kCodes;    // codewords of one matrix kind
constexpr int kTabFloats = 3 * kCodes * kTB;  // one kind's table of a slice: [stage][code][block]
constexpr int kBatch = 8;                 // rows a warp sums at once

// Launch geometry, the same on host and device.
struct RvqPlan {
  int S;          // input slices of H (gate|up)
  int R;          // gate|up rows of one token: k F + Fs
  int P, rpp;     // gate|up row parts per (token, kind, slice); rows per part (multiple of 8)
  int Sdr, Sds;   // down: slices of F and of Fs
  int Sdm;        // their maximum
  int Pd, rpd;    // down row parts per (token, entry, slice); rows per part (multiple of 8)
};

int cdiv(int a, int b) { return (a + b - 1) / b; }

RvqPlan rvq_plan(const LayerArgs& a, int num_sms) {
  RvqPlan p;
  const int slots = 2 * num_sms;  // two CTAs per SM
  p.R = a.k * a.F + a.Fs;
  p.S = cdiv(a.H / 8, kTB);
  p.P = std::max(1, std::min(slots / (2 * a.T * p.S), cdiv(p.R, kRvqWarps * kBatch)));
  p.rpp = cdiv(cdiv(p.R, p.P), kBatch) * kBatch;
  p.Sdr = cdiv(a.F / 8, kTB);
  p.Sds = a.Fs ? cdiv(a.Fs / 8, kTB) : 0;
  p.Sdm = std::max(p.Sdr, p.Sds);
  const int units = a.T * (a.k + (a.Fs ? 1 : 0)) * p.Sdm;
  p.Pd = std::max(1, std::min(slots / units, cdiv(a.H, kRvqWarps * kBatch)));
  p.rpd = cdiv(cdiv(a.H, p.Pd), kBatch) * kBatch;
  return p;
}

// The table, then 256 floats (the down kernel's h slice; the gate|up
// kernel's record pointers of the routed ranks and the shared expert).
size_t rvq_table_smem() { return kTabFloats * sizeof(float) + 256 * sizeof(float); }
static_assert((kMaxTopK + 1) * sizeof(void*) <= 256 * sizeof(float), "record table");

__device__ __forceinline__ float rvq_silu(float g) { return g / (1.0f + expf(-g)); }

// Lane j's entries T[stage][code][j] = <codeword(stage, code), v_j> of one
// kind's codebooks (book: 768 codewords as uint4 of 8 bf16), v_j the lane's
// 8 inputs; zero for lanes past the slice's nb blocks.  Warp w fills codes
// w, w + 16, ...: the codeword is one broadcast load, each lane's store its
// own bank.
__device__ __forceinline__ void build_table(const uint4* __restrict__ book, const float (&v)[8], bool act,
                                            float* __restrict__ T) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int q = warp; q < kKindWords; q += kRvqWarps) {
    const uint4 w = __ldg(book + q);
    float d = bf16lo(w.x) * v[0];
    d = fmaf(bf16hi(w.x), v[1], d), d = fmaf(bf16lo(w.y), v[2], d), d = fmaf(bf16hi(w.y), v[3], d);
    d = fmaf(bf16lo(w.z), v[4], d), d = fmaf(bf16hi(w.z), v[5], d), d = fmaf(bf16lo(w.w), v[6], d);
    d = fmaf(bf16hi(w.w), v[7], d);
    T[q * kTB + lane] = act ? d : 0.f;
  }
}

// Sums 8 per-lane row partials over the warp; lane L ends with the total of
// row L >> 2.
__device__ __forceinline__ float rvq_bfly8(const float (&p)[8], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float k[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b4 ? p[4 + i] : p[i], send = b4 ? p[i] : p[4 + i];
    k[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
  }
  float k2[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b3 ? k[2 + i] : k[i], send = b3 ? k[i] : k[2 + i];
    k2[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
  }
  float v = b2 ? k2[1] : k2[0];
  const float send = b2 ? k2[0] : k2[1];
  v += __shfl_xor_sync(0xFFFFFFFFu, send, 4);
  v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
  v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
  return v;
}

// Lane j's 3 code bytes of block j of 8 rows, whose slice chunks start at
// row0 + i * row_bytes (8-byte aligned): the aligned 32-bit word holding
// byte 3j and, for lanes whose bytes cross into the next word (j mod 4 in
// {1, 2}), that word too; both stay inside the 96-byte chunk.
struct CodeBatch {
  uint32_t lo[kBatch], hi[kBatch];
};

__device__ __forceinline__ void load_codes(const uint8_t* row0, size_t row_bytes, int lane, bool act,
                                           CodeBatch& c) {
  const int w = (3 * lane) >> 2;
  const bool two = ((lane & 3) == 1) || ((lane & 3) == 2);
#pragma unroll
  for (int i = 0; i < kBatch; ++i) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(row0 + i * row_bytes) + w;
    c.lo[i] = act ? __ldg(p) : 0u;
    c.hi[i] = (act && two) ? __ldg(p + 1) : 0u;
  }
}

// Per row of the batch: the sum of lane j's three table entries.  Entry
// (stage s, code c) of the lane sits c * 128 bytes into the stage's 32 KB.
__device__ __forceinline__ void lookup_batch(const CodeBatch& c, const float* __restrict__ T, int lane,
                                             float (&acc)[kBatch]) {
  const int sh = 8 * ((3 * lane) & 3);
  const char* Tl = reinterpret_cast<const char*>(T + lane);
#pragma unroll
  for (int i = 0; i < kBatch; ++i) {
    const uint32_t q = __funnelshift_r(c.lo[i], c.hi[i], sh);
    const float t0 = *reinterpret_cast<const float*>(Tl + ((q << 7) & 0x7F80u));
    const float t1 = *reinterpret_cast<const float*>(Tl + (kCodes * kTB * 4) + ((q >> 1) & 0x7F80u));
    const float t2 = *reinterpret_cast<const float*>(Tl + (2 * kCodes * kTB * 4) + ((q >> 9) & 0x7F80u));
    acc[i] = (t0 + t1) + t2;
  }
}

// Record of routed rank i of token t (through the cache's slot table when
// there is one: a slot outside the pool or holding another expert latches
// an error and is never read).
__device__ __forceinline__ const uint8_t* rvq_routed_record(const LayerArgs& a, int t, int i) {
  int e = a.ids[t * a.k + i];
  if (e < 0 || e >= a.E) latch_error(&a.ws.ctl[0], kErrRange), e = 0;
  int slot = e;
  if (a.slot_of) {
    slot = a.slot_of[e];
    if (slot < 0 || slot >= a.n_slots) latch_error(&a.ws.ctl[0], kErrResidency), slot = 0;
    else if (a.slot_tag && a.slot_tag[slot] != e) latch_error(&a.ws.ctl[0], kErrResidency);
  }
  return a.records + static_cast<size_t>(slot) * a.off_r.stride;
}

// Rows [r0, r1) of the CTA's row part, warp w taking batches w, w + 16, ...
// row_chunk(r) is row r's slice chunk (8 consecutive rows share a matrix);
// out(r) receives the row's partial sum.  The next batch's codes are loaded
// while the current one is looked up.
template <typename RowChunk, typename Out>
__device__ __forceinline__ void stream_rows(int r0, int r1, size_t row_bytes, int nbytes, bool act, const float* T,
                                            RowChunk row_chunk, Out out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int rb = r0 + warp * kBatch;
  if (rb >= r1) return;
  CodeBatch cur, nxt;
  load_codes(row_chunk(rb), row_bytes, lane, act, cur);
  (void)nbytes;
  for (; rb < r1; rb += kRvqWarps * kBatch) {
    const int rn = rb + kRvqWarps * kBatch;
    if (rn < r1) load_codes(row_chunk(rn), row_bytes, lane, act, nxt);
    float acc[kBatch];
    lookup_batch(cur, T, lane, acc);
    const float v = rvq_bfly8(acc, lane);
    if ((lane & 3) == 0 && rb + (lane >> 2) < r1) out(rb + (lane >> 2), v);
    cur = nxt;
  }
}

// grid T * 2 * S * P: CTA (token, kind, slice, part), kind 0 gate, 1 up.
// Partial sums to rvq_g (gate) / rvq_u (up) as [T][S][R].
__global__ void __launch_bounds__(kRvqThreads, 2) rvq_gateup_kernel(const __grid_constant__ LayerArgs a,
                                                                    const RvqPlan pl) {
  extern __shared__ __align__(16) float smem[];
  float* T = smem;
  int id = blockIdx.x;
  const int p = id % pl.P;
  id /= pl.P;
  const int s = id % pl.S;
  id /= pl.S;
  const int kind = id & 1, t = id >> 1;
  const int lane = threadIdx.x & 31;
  const int b0 = s * kTB, nb = min(kTB, a.H / 8 - b0);
  const bool act = lane < nb;
  pdl_launch_dependents();
  float v[8];
  {
    const uint4 w = act ? __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * a.H) + b0 + lane)
                        : make_uint4(0, 0, 0, 0);
    v[0] = bf16lo(w.x), v[1] = bf16hi(w.x), v[2] = bf16lo(w.y), v[3] = bf16hi(w.y);
    v[4] = bf16lo(w.z), v[5] = bf16hi(w.z), v[6] = bf16lo(w.w), v[7] = bf16hi(w.w);
  }
  build_table(reinterpret_cast<const uint4*>(a.cbs) + kind * kKindWords, v, act, T);
  pdl_wait();  // the router's ids (routed rows), and the previous step's readers of the partials
  const size_t row_bytes = static_cast<size_t>(a.H) / 8 * 3, o0 = static_cast<size_t>(s) * kTB * 3;
  // this kind's matrix of every routed rank, and of the shared expert (rank k)
  const uint8_t** mat = reinterpret_cast<const uint8_t**>(smem + kTabFloats);
  if (threadIdx.x < a.k)
    mat[threadIdx.x] = rvq_routed_record(a, t, threadIdx.x) + (kind ? a.off_r.up_codes : a.off_r.gate_codes) + o0;
  if (threadIdx.x == a.k && a.Fs) mat[a.k] = a.shared + (kind ? a.off_s.up_codes : a.off_s.gate_codes) + o0;
  __syncthreads();
  const int kF = a.k * a.F;
  float* part = (kind ? a.ws.rvq_u : a.ws.rvq_g) + (static_cast<size_t>(t) * pl.S + s) * pl.R;
  const int r0 = p * pl.rpp, r1 = min(pl.R, r0 + pl.rpp);
  stream_rows(
      r0, r1, row_bytes, 3 * nb, act, T,
      [&](int r) -> const uint8_t* {
        const int i = r < kF ? r / a.F : a.k, f = r < kF ? r - i * a.F : r - kF;
        return mat[i] + static_cast<size_t>(f) * row_bytes;
      },
      [&](int r, float val) { part[r] = val; });
}

// grid T * (k + 1) * Sdm * Pd: CTA (token, entry, slice of the entry's
// width, part); entry k is the shared expert.  h of the slice (SwiGLU of the
// gate|up partials added over the input slices in order), its table, then
// the down rows' partial sums to rvq_y as [T][k + 1][Sdm][H].
__global__ void __launch_bounds__(kRvqThreads, 2) rvq_down_kernel(const __grid_constant__ LayerArgs a,
                                                                  const RvqPlan pl) {
  extern __shared__ __align__(16) float smem[];
  float* T = smem;
  float* hs = smem + kTabFloats;  // the slice's 256 h values
  int id = blockIdx.x;
  const int p = id % pl.Pd;
  id /= pl.Pd;
  const int sd = id % pl.Sdm;
  id /= pl.Sdm;
  const int e = id % (a.k + 1), t = id / (a.k + 1);
  const bool sh = e == a.k;
  if (sh && a.Fs == 0) return;
  const int Fe = sh ? a.Fs : a.F;
  if (sd >= (sh ? pl.Sds : pl.Sdr)) return;
  const int lane = threadIdx.x & 31;
  const int b0 = sd * kTB, nb = min(kTB, Fe / 8 - b0);
  const bool act = lane < nb;
  pdl_launch_dependents();
  pdl_wait();  // the gate|up partials
  // h of the slice: thread i takes value i >> 1 of kind i & 1 (gate, up)
  const int rowb = sh ? a.k * a.F : e * a.F;
  for (int i = threadIdx.x; i < 2 * 256; i += kRvqThreads) {
    const int f = 8 * b0 + (i >> 1);
    float sum = 0.f;
    if (f < Fe) {
      const float* src = ((i & 1) ? a.ws.rvq_u : a.ws.rvq_g) + static_cast<size_t>(t) * pl.S * pl.R + rowb + f;
      for (int s = 0; s < pl.S; ++s) sum += __ldcg(src + static_cast<size_t>(s) * pl.R);
    }
    const float other = __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
    if ((i & 1) == 0) hs[i >> 1] = rvq_silu(sum) * other;
  }
  __syncthreads();
  float v[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) v[m] = act ? hs[8 * lane + m] : 0.f;
  build_table(reinterpret_cast<const uint4*>(a.cbs) + 2 * kKindWords, v, act, T);
  __syncthreads();
  const size_t row_bytes = static_cast<size_t>(Fe) / 8 * 3, o0 = static_cast<size_t>(b0) * 3;
  const uint8_t* codes = (sh ? a.shared + a.off_s.down_codes : rvq_routed_record(a, t, e) + a.off_r.down_codes) + o0;
  float* y = a.ws.rvq_y + ((static_cast<size_t>(t) * (a.k + 1) + e) * pl.Sdm + sd) * a.H;
  const int r0 = p * pl.rpd, r1 = min(a.H, r0 + pl.rpd);
  stream_rows(
      r0, r1, row_bytes, 3 * nb, act, T, [&](int r) { return codes + static_cast<size_t>(r) * row_bytes; },
      [&](int r, float val) { y[r] = val; });
}

// grid ceil(T H / 256): out = sum_i p_i y_i + y_shared, ranks in order, each
// y the sum of its slices in order.
__global__ void __launch_bounds__(256) rvq_combine_kernel(const __grid_constant__ LayerArgs a, const RvqPlan pl) {
  pdl_launch_dependents();
  pdl_wait();
  const size_t i = static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x;
  if (i >= static_cast<size_t>(a.T) * a.H) return;
  const int t = static_cast<int>(i / a.H), r = static_cast<int>(i - static_cast<size_t>(t) * a.H);
  const float* yt = a.ws.rvq_y + static_cast<size_t>(t) * (a.k + 1) * pl.Sdm * a.H + r;
  float acc = 0.f;
  for (int e = 0; e < a.k; ++e) {
    float y = 0.f;
    for (int sl = 0; sl < pl.Sdr; ++sl) y += __ldcg(yt + (static_cast<size_t>(e) * pl.Sdm + sl) * a.H);
    acc = fmaf(a.weights[t * a.k + e], y, acc);
  }
  if (a.Fs) {
    float y = 0.f;
    for (int sl = 0; sl < pl.Sds; ++sl) y += __ldcg(yt + (static_cast<size_t>(a.k) * pl.Sdm + sl) * a.H);
    acc += y;
  }
  a.out_bf16[i] = f32_to_bf16_rne(acc);
  if (a.out_f32) a.out_f32[i] = acc;
}

cudaError_t launch_rvq(const void* fn, int grid, int block, size_t smem, cudaStream_t st, bool pdl,
                       const LayerArgs& a, const RvqPlan& pl) {
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
  void* args[] = {const_cast<LayerArgs*>(&a), const_cast<RvqPlan*>(&pl)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t mark_rvq(const LayerArgs& a, int i, cudaStream_t st) {
  return a.prof_on ? cudaEventRecord(static_cast<cudaEvent_t>(a.prof[i]), st) : cudaSuccess;
}

}  // namespace

size_t rvq_smem_need(const LayerArgs&) { return rvq_table_smem(); }

// Bytes of the residual-VQ partial sums for T tokens: gate and up [T][S][R],
// down [T][k + 1][Sdm][H] (the workspace carve).
size_t rvq_partial_floats(int H, int k, int F, int Fs, int T, int which) {
  const int S = cdiv(H / 8, kTB), R = k * F + Fs;
  const int Sdm = std::max(cdiv(F / 8, kTB), Fs ? cdiv(Fs / 8, kTB) : 0);
  return which < 2 ? static_cast<size_t>(T) * S * R : static_cast<size_t>(T) * (k + 1) * Sdm * H;
}

cudaError_t set_rvq_attributes(int smem_optin) {
  (void)smem_optin;
  const int bytes = static_cast<int>(rvq_table_smem());
  cudaError_t e = cudaFuncSetAttribute(rvq_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e ? e : cudaFuncSetAttribute(rvq_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// gate|up, down and the combine for every token at once, after a router
// launch of the same step (the expert cache runs them after its copies).
cudaError_t launch_rvq_experts(const LayerArgs& a, int num_sms, cudaStream_t st) {
  const bool pdl = !a.prof_on;
  const RvqPlan pl = rvq_plan(a, num_sms);
  const int gu = a.T * 2 * pl.S * pl.P, dn = a.T * (a.k + 1) * pl.Sdm * pl.Pd;
  const int cb = cdiv(a.T * a.H, 256);
  cudaError_t e;
  if ((e = launch_rvq((const void*)rvq_gateup_kernel, gu, kRvqThreads, rvq_table_smem(), st, pdl, a, pl)) ||
      (e = mark_rvq(a, 2, st)) ||
      (e = launch_rvq((const void*)rvq_down_kernel, dn, kRvqThreads, rvq_table_smem(), st, pdl, a, pl)) ||
      (e = launch_rvq((const void*)rvq_combine_kernel, cb, 256, 0, st, pdl, a, pl)))
    return e;
  return cudaSuccess;
}

// The router, then gate|up, down and the combine for every token at once.
// Profile events: before the router, before gate|up, before down, after the
// combine.
cudaError_t launch_decode_rvq(const LayerArgs& a, int num_sms, cudaStream_t st) {
  cudaError_t e;
  if ((e = mark_rvq(a, 0, st)) || (e = launch_decode_router(a, num_sms, st)) || (e = mark_rvq(a, 1, st)) ||
      (e = launch_rvq_experts(a, num_sms, st)))
    return e;
  return mark_rvq(a, 3, st);
}

}  // namespace moe
