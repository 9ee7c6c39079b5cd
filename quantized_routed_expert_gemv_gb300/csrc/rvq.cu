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
// cut into slices of 64 blocks (512 inputs) and a CTA tabulates one slice of
// one matrix kind: 192 KB of shared memory laid out [stage][code][block],
// one 256-byte row per (stage, code).  Lane j owns two blocks of the slice
// for every row, 2j and 2j + 1, and looks them up in turn: lanes 0-15 take
// 2j first, lanes 16-31 2j + 1, so the first lookup of a warp hits the even
// banks from its low half and the odd banks from its high half, the second
// the other way round, and every lookup instruction is one conflict-free
// wavefront whatever the codes are.  A lane's 6 code bytes of a row sit in
// two aligned 32-bit words; one byte permute puts them in lookup order and
// one more per lookup builds the table offset (stage << 16 | code << 8 |
// 4 * block).  A warp takes 8 rows at a time and sums each row over its
// lanes with one 8-row butterfly.  Partial sums per slice land in the
// workspace; later kernels add them in a fixed order.
//
// Each kernel runs one CTA per SM over the 8-row batches of all its units (a
// unit: one table, i.e. one token, matrix kind and slice).  With at least two
// CTAs per unit every CTA takes a contiguous part of one unit and builds one
// table; otherwise the flat list of batches is cut into equal contiguous
// shares and a CTA builds a few tables.  One launch of each serves every
// token of the step:
//   rvq_gateup_kernel   units (token, kind, slice): gate or up partial sums of
//                       the token's routed experts and the shared expert; the
//                       CTA's first table is built before the wait for the
//                       router, so it overlaps the router
//   rvq_down_kernel     units (token, entry, slice of F): h of the slice from
//                       the gate|up partials (SwiGLU), its table, then the
//                       down partial sums
//   rvq_combine_kernel  out = sum_i p_i y_i + y_shared, bf16 and f32
#include <algorithm>
#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

cudaError_t launch_decode_router(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_b1_router(const LayerArgs& a, int num_sms, cudaStream_t st);

namespace {

constexpr int kRvqThreads = 512;            // 16 warps
constexpr int kRvqWarps = kRvqThreads / 32;
constexpr int kSB = 64;                     // blocks of 8 inputs per slice: two per lane
constexpr int kCodes = 256;                 // codewords per stage
constexpr int kKindWords = 3 * kCodes;      // codewords of one matrix kind
constexpr int kRowBytes = kSB * 4;          // one (stage, code) row of the table
constexpr int kTabBytes = 3 * kCodes * kRowBytes;  // 196,608: [stage][code][block]
constexpr int kBatch = 8;                   // rows a warp sums at once
constexpr int kChunkBytes = 3 * kSB;        // a row's code bytes of one slice
// The shared address at which dynamic shared memory starts in a kernel with
// no static shared memory on this part (after the CTA's reserved 1 KB).  The
// lookups of a table there carry its address as an immediate; a table at
// any other address takes the same lookups with one add each.
constexpr int kDynSmemBase = 1024;

// Launch geometry, the same on host and device.
struct RvqPlan {
  int S;          // input slices of H (gate|up)
  int R;          // gate|up rows of one token: k F + Fs
  int Sdr, Sds;   // down: slices of F and of Fs
  int Sdm;        // their maximum
  int upt;        // down units of one token: k Sdr + Sds
  long long gu_batches, dn_batches;  // 8-row batches of all units
  int grid;       // CTAs of each kernel (one per SM)
};

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

RvqPlan rvq_plan(const LayerArgs& a, int num_sms) {
  RvqPlan p;
  p.R = a.k * a.F + a.Fs;
  p.S = cdiv(a.H / 8, kSB);
  p.Sdr = cdiv(a.F / 8, kSB);
  p.Sds = a.Fs ? cdiv(a.Fs / 8, kSB) : 0;
  p.Sdm = std::max(p.Sdr, p.Sds);
  p.upt = a.k * p.Sdr + p.Sds;
  p.gu_batches = static_cast<long long>(a.T) * 2 * p.S * cdiv(p.R, kBatch);
  p.dn_batches = static_cast<long long>(a.T) * p.upt * cdiv(a.H, kBatch);
  p.grid = std::max(1, num_sms);
  return p;
}

// The table, then the matrix kind's codebooks (768 codewords, 12 KB), then
// 2 KB: the down kernel's h slice (512 floats) or the gate|up kernel's record
// pointers of the routed ranks and the shared expert.
constexpr int kBookBytes = kKindWords * 16;
size_t rvq_table_smem() { return kTabBytes + kBookBytes + 512 * sizeof(float); }
static_assert((kMaxTopK + 1) * sizeof(void*) <= 512 * sizeof(float), "record table");

__device__ __forceinline__ float rvq_silu(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// The same with a selector known at compile time (an immediate operand).
template <uint32_t SEL>
__device__ __forceinline__ uint32_t prmt_i(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "n"(SEL));
  return d;
}

// The kind's 768 codewords (uint4 of 8 bf16 each) into shared memory, every
// load of the CTA in flight at once; the caller synchronises before use.
__device__ __forceinline__ void stage_book(const uint4* __restrict__ book, uint4* __restrict__ sbook) {
  for (int q = threadIdx.x; q < kKindWords; q += kRvqThreads) sbook[q] = __ldg(book + q);
}

// Lane j's entries T[stage][code][2j], T[...][2j + 1] = <codeword(stage,
// code), v_b> of one kind's codebooks (sbook: the 768 codewords in shared
// memory), vA/vB the lane's two blocks of 8 inputs; zero for lanes past the
// slice's nb blocks.  Warp w fills codewords w, w + 16, ...: the codeword is
// one broadcast read, and the warp's 32 float2 stores fill one table row.
__device__ __forceinline__ void build_table(const uint4* __restrict__ sbook, const float (&vA)[8],
                                            const float (&vB)[8], bool act, uint8_t* __restrict__ T) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int q = warp; q < kKindWords; q += kRvqWarps) {
    const uint4 w = sbook[q];
    const float c[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                        bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
    float dA = c[0] * vA[0], dB = c[0] * vB[0];
#pragma unroll
    for (int m = 1; m < 8; ++m) dA = fmaf(c[m], vA[m], dA), dB = fmaf(c[m], vB[m], dB);
    *reinterpret_cast<float2*>(T + q * kRowBytes + 8 * lane) = act ? make_float2(dA, dB) : make_float2(0.f, 0.f);
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

// A lane's per-row constants.  Its 6 code bytes of a row (blocks 2j and
// 2j + 1, 3 stage bytes each) start d = 6j mod 4 bytes into the aligned word
// pair (w0, w1) at byte 4 * wo of the slice chunk.  sel_lo / sel_hi permute
// them so that lo holds the first-looked-up block's 3 bytes and the other
// block's first byte, hi the other block's last two; base[i] holds
// stage << 16 | 4 * block for lookup i (first block's stages 0-2, then the
// second block's).
struct Lane {
  int wo;
  uint32_t sel_lo, sel_hi;
  uint32_t base[6];
  bool act;
};

__device__ __forceinline__ Lane lane_consts(int lane, int nb) {
  Lane L;
  const int d = (6 * lane) & 3;
  L.wo = (6 * lane) >> 2;
  L.act = 2 * lane < nb;
  if (!L.act) L.wo = 0;  // reads valid bytes of the row; its table entries are zero
  const bool hi16 = lane >= 16;
  const int first = hi16 ? 2 * lane + 1 : 2 * lane, second = hi16 ? 2 * lane : 2 * lane + 1;
  // bytes of block 2j: d .. d + 2; of block 2j + 1: d + 3 .. d + 5
  const int f0 = hi16 ? d + 3 : d, s0 = hi16 ? d : d + 3;
  L.sel_lo = static_cast<uint32_t>(f0 | (f0 + 1) << 4 | (f0 + 2) << 8 | s0 << 12);
  L.sel_hi = static_cast<uint32_t>((s0 + 1) | (s0 + 2) << 4 | (s0 + 1) << 8 | (s0 + 1) << 12);
#pragma unroll
  for (int st = 0; st < 3; ++st) {
    L.base[st] = static_cast<uint32_t>(st << 16 | 4 * first);
    L.base[3 + st] = static_cast<uint32_t>(st << 16 | 4 * second);
  }
  return L;
}

struct CodeBatch {
  uint32_t w0[kBatch], w1[kBatch];
  const uint8_t* row0;  // the batch's first slice chunk
};

// Lane's code words of row i of a batch whose slice chunks start at row0 +
// i * row_bytes.  Both words of a row go out together and through L1, so the
// second one meets the first one's sectors on the SM.  Every lane loads
// (a lane past the slice's blocks reads the row's first word pair), so the
// loads need no predicate.
__device__ __forceinline__ void load_row(const uint8_t* row0, size_t row_bytes, const Lane& L, int i,
                                         CodeBatch& c) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(row0 + i * row_bytes) + L.wo;
  c.w0[i] = __ldca(p);
  c.w1[i] = __ldca(p + 1);
}

__device__ __forceinline__ void load_codes(const uint8_t* row0, size_t row_bytes, const Lane& L, CodeBatch& c) {
  c.row0 = row0;
#pragma unroll
  for (int i = 0; i < kBatch; ++i) load_row(row0, row_bytes, L, i, c);
}

// One table entry at shared offset `off` from the table.  kBase >= 0: the
// table's shared address, known at compile time, goes into the load as an
// immediate; otherwise tb is added.
template <int kBase>
__device__ __forceinline__ float tab(uint32_t off, uint32_t tb) {
  float v;
  if constexpr (kBase >= 0)
    asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(off), "n"(kBase));
  else
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(off + tb));
  return v;
}

__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  unsigned long long d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Row i's six lookups, packed with row i + 1's (lane-wise pairs of f32).
template <int kBase>
__device__ __forceinline__ void lookup_row(uint32_t lo, uint32_t hi, const Lane& L, uint32_t tb, float (&v)[6]) {
  // offset = stage << 16 | code << 8 | 4 * block: byte 0 and 2 from base, byte 1 the code
  v[0] = tab<kBase>(prmt_i<0x7604u>(lo, L.base[0]), tb);
  v[1] = tab<kBase>(prmt_i<0x7614u>(lo, L.base[1]), tb);
  v[2] = tab<kBase>(prmt_i<0x7624u>(lo, L.base[2]), tb);
  v[3] = tab<kBase>(prmt_i<0x7634u>(lo, L.base[3]), tb);
  v[4] = tab<kBase>(prmt_i<0x7604u>(hi, L.base[4]), tb);
  v[5] = tab<kBase>(prmt_i<0x7614u>(hi, L.base[5]), tb);
}

// Per row of the batch: the sum of the lane's six table entries, two rows
// at a time in packed f32 pairs (each row's sum in the order ((a0 + a1) +
// a2) + ((b0 + b1) + b2)).  Once a row's words are used, the same registers
// take that row of the batch at `next`, so a warp keeps about two batches of
// code loads in flight with one spare register set.  With no batch left to
// fetch, `next` is the batch's own rows again (cached, and never looked up),
// which keeps the loop free of branches.
template <int kBase>
__device__ __forceinline__ void lookup_batch(CodeBatch& c, uint32_t tb, const Lane& L, const uint8_t* next,
                                             size_t row_bytes, float (&acc)[kBatch]) {
  c.row0 = next;
#pragma unroll
  for (int i = 0; i < kBatch; i += 2) {
    float v[6], w[6];
    {
      const uint32_t lo = prmt(c.w0[i], c.w1[i], L.sel_lo), hi = prmt(c.w0[i], c.w1[i], L.sel_hi);
      load_row(next, row_bytes, L, i, c);
      lookup_row<kBase>(lo, hi, L, tb, v);
    }
    {
      const uint32_t lo = prmt(c.w0[i + 1], c.w1[i + 1], L.sel_lo), hi = prmt(c.w0[i + 1], c.w1[i + 1], L.sel_hi);
      load_row(next, row_bytes, L, i + 1, c);
      lookup_row<kBase>(lo, hi, L, tb, w);
    }
    const unsigned long long a = add2(add2(pack2(v[0], w[0]), pack2(v[1], w[1])), pack2(v[2], w[2]));
    const unsigned long long b = add2(add2(pack2(v[3], w[3]), pack2(v[4], w[4])), pack2(v[5], w[5]));
    const unsigned long long r = add2(a, b);
    asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[i]), "=f"(acc[i + 1]) : "l"(r));
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

// Batches [b0, b1) of a unit (rows 8 b .. 8 b + 7, clipped at nrows), warp
// w taking b0 + w, b0 + w + 16, ...  Cur is a row cursor: at(b) places it on
// batch b's first row, then next() steps it 16 batches on; ptr() is that
// row's slice chunk (8 consecutive rows share a matrix).  out(r) receives
// row r's partial sum.  Two register sets alternate: while one batch is
// looked up its registers are refilled with the batch two ahead, and the
// other set's loads (the next batch) are in flight.  A second cursor runs
// kPfAhead batches ahead and prefetches their chunks into L2 (a chunk of
// `chunk` bytes spans at most two 128-byte lines: lane 2i takes row i's
// first byte, lane 2i + 1 the byte 128 on, clipped to the chunk).
constexpr int kPfAhead = 4;
template <int kBase, typename Cur, typename Out>
__device__ __forceinline__ void stream_batches(long long b0, long long b1, int nrows, size_t row_bytes, int chunk,
                                               const Lane& L, uint32_t tb, Cur cur, Out out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long b = b0 + warp;
  if (b >= b1) return;
  constexpr int W = kRvqWarps;
  const size_t pf_off = static_cast<size_t>(lane >> 1) * row_bytes + ((lane & 1) ? min(128, chunk - 1) : 0);
  Cur pf = cur;
  auto prefetch = [&](long long bb) {  // pf on batch bb
    if (bb < b1 && lane < 2 * kBatch) asm volatile("prefetch.global.L2 [%0];" ::"l"(pf.ptr() + pf_off));
    pf.next();
  };
  pf.at(static_cast<int>(b + 2 * W) * kBatch);
#pragma unroll
  for (int j = 2; j < kPfAhead; ++j) prefetch(b + j * W);
  CodeBatch A, B;
  cur.at(static_cast<int>(b) * kBatch);
  load_codes(cur.ptr(), row_bytes, L, A);
  cur.next();
  if (b + W < b1) load_codes(cur.ptr(), row_bytes, L, B);
  cur.next();  // on batch b + 2W: the refill of the first set
  auto one = [&](CodeBatch& c, long long bb) {
    float acc[kBatch];
    prefetch(bb + kPfAhead * W);
    const uint8_t* next = bb + 2 * W < b1 ? cur.ptr() : c.row0;
    lookup_batch<kBase>(c, tb, L, next, row_bytes, acc);
    cur.next();
    const float v = rvq_bfly8(acc, lane);
    const int r = static_cast<int>(bb) * kBatch + (lane >> 2);
    if ((lane & 3) == 0 && r < nrows) out(r, v);
  };
  for (;;) {
    one(A, b);
    if ((b += W) >= b1) break;
    one(B, b);
    if ((b += W) >= b1) break;
  }
}

// Row cursor over the rows of one matrix (the down matrix of an entry).
struct FlatCur {
  const uint8_t* base;
  size_t row_bytes;
  int r;
  __device__ __forceinline__ void at(int r0) { r = r0; }
  __device__ __forceinline__ void next() { r += kRvqWarps * kBatch; }
  __device__ __forceinline__ const uint8_t* ptr() const { return base + static_cast<size_t>(r) * row_bytes; }
};

// Row cursor over the gate (or up) rows of a token: k routed matrices of F
// rows, then the shared expert's Fs rows (mat[i] the slice chunk of matrix
// i's first row).  Steps without division once placed.
struct GuCur {
  const uint8_t* const* mat;
  size_t row_bytes;
  int k, F, Fs, i, f;
  __device__ __forceinline__ void at(int r) {
    i = r / F;
    if (i > k) i = k;
    f = r - i * F;
    norm();
  }
  __device__ __forceinline__ void norm() {
    while (i < k && f >= F) f -= F, ++i;
  }
  __device__ __forceinline__ void next() {
    f += kRvqWarps * kBatch;
    norm();
  }
  __device__ __forceinline__ const uint8_t* ptr() const {
    // past the last row (no batch reads it): a valid address all the same
    const int ii = i > k ? k : i, ff = (i == k && f >= Fs) ? 0 : f;
    return mat[ii] + static_cast<size_t>(ff) * row_bytes;
  }
};

// This CTA's share [lo, hi) of n batches over `grid` CTAs.
__device__ __forceinline__ void cta_share(long long n, int grid, long long& lo, long long& hi) {
  lo = n * blockIdx.x / grid;
  hi = n * (blockIdx.x + 1) / grid;
}

// With at least two CTAs per unit, every CTA takes a part of exactly one
// unit (units split into G / U or G / U + 1 equal parts), so no CTA builds
// two tables; otherwise (one part per unit would leave whole units to
// single CTAs beside halves) the flat share.
__device__ __forceinline__ void unit_share(int units, int nbu, int grid, long long& lo, long long& hi) {
  if (2 * units > grid) {
    cta_share(static_cast<long long>(units) * nbu, grid, lo, hi);
    return;
  }
  const int q = grid / units, r = grid % units, c = blockIdx.x;
  int u, part, parts;
  if (c < r * (q + 1)) {
    u = c / (q + 1), part = c % (q + 1), parts = q + 1;
  } else {
    const int c2 = c - r * (q + 1);
    u = r + c2 / q, part = c2 % q, parts = q;
  }
  const long long u0 = static_cast<long long>(u) * nbu;
  lo = u0 + static_cast<long long>(nbu) * part / parts;
  hi = u0 + static_cast<long long>(nbu) * (part + 1) / parts;
}

// Units (token, kind, slice), kind 0 gate, 1 up, each cdiv(R, 8) batches of
// the rows of the token's k routed experts then the shared expert.  Partial
// sums to rvq_g (gate) / rvq_u (up) as [T][S][R].
__global__ void __launch_bounds__(kRvqThreads, 1) rvq_gateup_kernel(const __grid_constant__ LayerArgs a,
                                                                    const RvqPlan pl) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* T = smem;
  const uint32_t tb = static_cast<uint32_t>(__cvta_generic_to_shared(T));
  uint4* sbook = reinterpret_cast<uint4*>(smem + kTabBytes);
  const uint8_t** mat = reinterpret_cast<const uint8_t**>(smem + kTabBytes + kBookBytes);
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();
  const int nbu = cdiv(pl.R, kBatch);  // batches per unit
  long long lo, hi;
  unit_share(a.T * 2 * pl.S, nbu, gridDim.x, lo, hi);
  const size_t row_bytes = static_cast<size_t>(a.H) / 8 * 3;
  bool routed = false;
  for (long long u = lo / nbu; u * nbu < hi; ++u) {
    const int s = static_cast<int>(u % pl.S), kind = static_cast<int>((u / pl.S) & 1),
              t = static_cast<int>(u / (2 * pl.S));
    const int nb = min(kSB, a.H / 8 - s * kSB);
    const Lane L = lane_consts(lane, nb);
    float vA[8], vB[8];
    {
      const uint4* xp = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * a.H) + s * kSB + 2 * lane;
      const uint4 wa = L.act ? __ldg(xp) : make_uint4(0, 0, 0, 0), wb = L.act ? __ldg(xp + 1) : make_uint4(0, 0, 0, 0);
      const uint32_t A[4] = {wa.x, wa.y, wa.z, wa.w}, B[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        vA[2 * m] = bf16lo(A[m]), vA[2 * m + 1] = bf16hi(A[m]);
        vB[2 * m] = bf16lo(B[m]), vB[2 * m + 1] = bf16hi(B[m]);
      }
    }
    __syncthreads();  // the previous unit's lookups and table builders are done
    stage_book(reinterpret_cast<const uint4*>(a.cbs) + kind * kKindWords, sbook);
    __syncthreads();
    build_table(sbook, vA, vB, L.act, T);
    if (!routed) {
      pdl_wait();  // the router's ids (routed rows), and the previous step's readers of the partials
      routed = true;
    }
    // this kind's matrix of every routed rank, and of the shared expert (rank k)
    const size_t o0 = static_cast<size_t>(s) * kChunkBytes;
    if (threadIdx.x < a.k)
      mat[threadIdx.x] = rvq_routed_record(a, t, threadIdx.x) + (kind ? a.off_r.up_codes : a.off_r.gate_codes) + o0;
    if (threadIdx.x == a.k && a.Fs) mat[a.k] = a.shared + (kind ? a.off_s.up_codes : a.off_s.gate_codes) + o0;
    __syncthreads();
    float* part = (kind ? a.ws.rvq_u : a.ws.rvq_g) + (static_cast<size_t>(t) * pl.S + s) * pl.R;
    const long long u0 = u * nbu;
    GuCur gc;
    gc.mat = mat, gc.row_bytes = row_bytes, gc.k = a.k, gc.F = a.F, gc.Fs = a.Fs;
    const auto out = [&](int r, float val) { part[r] = val; };
    if (tb == kDynSmemBase)
      stream_batches<kDynSmemBase>(max(lo, u0) - u0, min(hi, u0 + nbu) - u0, pl.R, row_bytes, 3 * nb, L, tb, gc, out);
    else
      stream_batches<-1>(max(lo, u0) - u0, min(hi, u0 + nbu) - u0, pl.R, row_bytes, 3 * nb, L, tb, gc, out);
  }
  if (!routed) pdl_wait();
}

// Units (token, entry, slice of the entry's width): entry i < k routed rank
// i (Sdr slices each), then the shared expert (Sds slices); each cdiv(H, 8)
// batches of down rows.  h of the slice (SwiGLU of the gate|up partials
// added over the input slices in order), its table, then the down rows'
// partial sums to rvq_y as [T][k + 1][Sdm][H].
__global__ void __launch_bounds__(kRvqThreads, 1) rvq_down_kernel(const __grid_constant__ LayerArgs a,
                                                                  const RvqPlan pl) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* T = smem;
  const uint32_t tb = static_cast<uint32_t>(__cvta_generic_to_shared(T));
  uint4* sbook = reinterpret_cast<uint4*>(smem + kTabBytes);
  float* hs = reinterpret_cast<float*>(smem + kTabBytes + kBookBytes);  // the slice's 512 h values
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();
  // the down codebooks are the same for every unit: staged once
  stage_book(reinterpret_cast<const uint4*>(a.cbs) + 2 * kKindWords, sbook);
  pdl_wait();  // the gate|up partials
  const int nbu = cdiv(a.H, kBatch);
  long long lo, hi;
  unit_share(a.T * pl.upt, nbu, gridDim.x, lo, hi);
  for (long long u = lo / nbu; u * nbu < hi; ++u) {
    const int t = static_cast<int>(u / pl.upt), rem = static_cast<int>(u % pl.upt);
    const bool sh = rem >= a.k * pl.Sdr;
    const int e = sh ? a.k : rem / pl.Sdr, sd = sh ? rem - a.k * pl.Sdr : rem % pl.Sdr;
    const int Fe = sh ? a.Fs : a.F;
    const int nb = min(kSB, Fe / 8 - sd * kSB);
    const Lane L = lane_consts(lane, nb);
    __syncthreads();  // the previous unit's lookups and h readers are done
    // h of the slice: thread i takes value i of gate (sum over the S input
    // slices in order) and the same value of up
    const int rowb = sh ? a.k * a.F : e * a.F;
    {
      const int i = threadIdx.x, f = 8 * kSB * sd + i;
      float g = 0.f, up = 0.f;
      if (f < Fe) {
        const size_t o = static_cast<size_t>(t) * pl.S * pl.R + rowb + f;
#pragma unroll 8
        for (int s = 0; s < pl.S; ++s) {
          g += __ldcg(a.ws.rvq_g + o + static_cast<size_t>(s) * pl.R);
          up += __ldcg(a.ws.rvq_u + o + static_cast<size_t>(s) * pl.R);
        }
      }
      hs[i] = rvq_silu(g) * up;
    }
    __syncthreads();
    float vA[8], vB[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) vA[m] = hs[16 * lane + m], vB[m] = hs[16 * lane + 8 + m];
    build_table(sbook, vA, vB, L.act, T);
    __syncthreads();
    const size_t row_bytes = static_cast<size_t>(Fe) / 8 * 3, o0 = static_cast<size_t>(sd) * kChunkBytes;
    const uint8_t* codes = (sh ? a.shared + a.off_s.down_codes : rvq_routed_record(a, t, e) + a.off_r.down_codes) + o0;
    float* y = a.ws.rvq_y + ((static_cast<size_t>(t) * (a.k + 1) + e) * pl.Sdm + sd) * a.H;
    const long long u0 = u * nbu;
    FlatCur fc;
    fc.base = codes, fc.row_bytes = row_bytes;
    const auto out = [&](int r, float val) { y[r] = val; };
    if (tb == kDynSmemBase)
      stream_batches<kDynSmemBase>(max(lo, u0) - u0, min(hi, u0 + nbu) - u0, a.H, row_bytes, 3 * nb, L, tb, fc, out);
    else
      stream_batches<-1>(max(lo, u0) - u0, min(hi, u0 + nbu) - u0, a.H, row_bytes, 3 * nb, L, tb, fc, out);
  }
}

// out = sum_i p_i y_i + y_shared, each y the sum of its slices in order.
// A CTA takes 32 consecutive outputs of one token; its 8 warps split the
// ranks (warp g: ranks g, g + 8, ..., the shared expert in warp 0), so each
// thread has few dependent loads, and the warps' sums are added in warp
// order: the same order for every launch.
constexpr int kCombThreads = 256, kCombOut = 32, kCombGroups = kCombThreads / kCombOut;
__global__ void __launch_bounds__(kCombThreads) rvq_combine_kernel(const __grid_constant__ LayerArgs a,
                                                                   const RvqPlan pl) {
  __shared__ float red[kCombGroups][kCombOut];
  pdl_launch_dependents();
  pdl_wait();
  const int per_t = (a.H + kCombOut - 1) / kCombOut;
  const int t = blockIdx.x / per_t, r = (blockIdx.x % per_t) * kCombOut + (threadIdx.x & 31);
  const int g = threadIdx.x >> 5;
  float acc = 0.f;
  if (r < a.H) {
    const float* yt = a.ws.rvq_y + static_cast<size_t>(t) * (a.k + 1) * pl.Sdm * a.H + r;
    for (int e = g; e < a.k; e += kCombGroups) {
      const float* ye = yt + static_cast<size_t>(e) * pl.Sdm * a.H;
      float y = 0.f;
      for (int sl = 0; sl < pl.Sdr; ++sl) y += __ldcg(ye + static_cast<size_t>(sl) * a.H);
      acc = fmaf(a.weights[t * a.k + e], y, acc);
    }
    if (g == 0 && a.Fs) {
      const float* ye = yt + static_cast<size_t>(a.k) * pl.Sdm * a.H;
      float y = 0.f;
      for (int sl = 0; sl < pl.Sds; ++sl) y += __ldcg(ye + static_cast<size_t>(sl) * a.H);
      acc += y;
    }
  }
  red[g][threadIdx.x & 31] = acc;
  __syncthreads();
  if (g == 0 && r < a.H) {
    float out = red[0][threadIdx.x];
    for (int j = 1; j < kCombGroups; ++j) out += red[j][threadIdx.x];
    const size_t i = static_cast<size_t>(t) * a.H + r;
    a.out_bf16[i] = f32_to_bf16_rne(out);
    if (a.out_f32) a.out_f32[i] = out;
  }
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
  const int S = cdiv(H / 8, kSB), R = k * F + Fs;
  const int Sdm = std::max(cdiv(F / 8, kSB), Fs ? cdiv(Fs / 8, kSB) : 0);
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
  const int cb = a.T * cdiv(a.H, kCombOut);
  cudaError_t e;
  if ((e = launch_rvq((const void*)rvq_gateup_kernel, pl.grid, kRvqThreads, rvq_table_smem(), st, pdl, a, pl)) ||
      (e = mark_rvq(a, 2, st)) ||
      (e = launch_rvq((const void*)rvq_down_kernel, pl.grid, kRvqThreads, rvq_table_smem(), st, pdl, a, pl)) ||
      (e = launch_rvq((const void*)rvq_combine_kernel, cb, kCombThreads, 0, st, pdl, a, pl)))
    return e;
  return cudaSuccess;
}

// The router (the single-token one, with its block-wide top-k, for one
// token), then gate|up, down and the combine for every token at once.
// Profile events: before the router, before gate|up, before down, after the
// combine.
cudaError_t launch_decode_rvq(const LayerArgs& a, int num_sms, cudaStream_t st) {
  cudaError_t e;
  if ((e = mark_rvq(a, 0, st)) ||
      (e = a.T == 1 ? launch_b1_router(a, num_sms, st) : launch_decode_router(a, num_sms, st)) ||
      (e = mark_rvq(a, 1, st)) ||
      (e = launch_rvq_experts(a, num_sms, st)))
    return e;
  return mark_rvq(a, 3, st);
}

}  // namespace moe
