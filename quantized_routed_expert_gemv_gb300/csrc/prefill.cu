// prefill.cu -- a prefill chunk (T <= 128 tokens) on the fifth-generation
// tensor cores.
//
// TurboFieldfare page, section "Token üretim süreci": prompt prefill runs in
// chunks of at most 128 tokens so that one fetched expert serves several
// rows.  With up to 128 tokens per expert the expert FFN is a small dense
// contraction: each expert's 4-bit weights are read from HBM once per chunk
// and multiplied against all of its tokens on the tensor cores.
//
// Kernels, in stream order (T >= kPrefillTcMin and H, F, Fs multiples of 128;
// other chunks run the decode kernels):
//   router          decode.cu's router for T tokens: logits, top-k, weights,
//                   grouping by expert.
//   pf_pack_kernel  CTAs over (entry, 16 packed rows) (shared expert, then active experts):
//                   splits the entry's tokens into blocks of <= 64, writes the
//                   block table, the activations in the tensor core's
//                   core-matrix order (see below) and their per-group sums.
//   pf_gemm_kernel<0>  gate|up: items = (block, 64 gate rows + the same 64 up
//                   rows); D = [W_g; W_u] x^T, then SwiGLU, h packed as bf16
//                   hi + lo for the down GEMM.
//   pf_gemm_kernel<1>  down: items = (block, 128 rows of H); y = W_d h.
//   pf_combine_kernel  out = y_shared + sum_i p_i y_{e_i}, fixed order.
//
// Exact 4-bit weights on the tensor cores.  A weight is s*q + b (s, b bf16
// per group of 64 along K, q in 0..15).  The A operand holds the code q
// itself as bf16: four masks turn a 32-bit word of 8 codes into bf16 pairs
// 128 + q (bits 0x4300 | q), and one exact bf16x2 FMA per pair removes the
// 128.  Each group of 64 K-values accumulates into its own TMEM columns, and
// the epilogue applies  s * D_g + b * X_g  with X_g the group sum of the
// activations (fp32), so no weight is rounded.  The masks yield the codes of
// a word in the order 0,4,1,5,2,6,3,7; the activations are packed in the
// same order, so the contraction is unchanged.
// The down GEMM's h is fp32; it is split into bf16 hi + lo (two MMAs into
// the same accumulator), error about 2^-17 relative.
//
// Operands: A (the dequantised codes) lives in TMEM, row m in lane m, two
// bf16 per 32-bit column in K order; B (activations) in shared memory, no
// swizzle, K-major core matrices of 8 rows x 16 bytes: within a 128-K chunk,
// core (k8, r8) sits at (k8 * R8 + r8) * 128 bytes (R8 = rows / 8), so the
// descriptor's leading offset is the K-direction core stride (R8 * 128) and
// its stride offset the 8-row stride (128).
//
// Warp roles of pf_gemm_kernel (12 warps, one CTA per SM, persistent over
// items): warps 0-3 epilogue (TMEM lanes 32*w.., all of a block's columns),
// warps 4-7 dequantise codes into TMEM (lanes 32*(w-4)..), warp 8 streams
// the activation (B) chunks, warp 9 streams codes (tiled TMA loads) and
// group sums, warps 10-11 issue the MMAs (alternate chunks; warp 10 also
// allocates TMEM).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace moe {

cudaError_t launch_decode(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_decode_router(const LayerArgs& a, int num_sms, cudaStream_t st);

constexpr int kPrefillTcMin = 32;  // smaller chunks: the decode kernels
constexpr unsigned kAllLanes = 0xFFFFFFFFu;
constexpr int kBlkTokens = 64;     // tokens per block (N of the MMA <= 64)

__host__ __device__ inline int round16(int v) { return (v + 15) & ~15; }
// Chunks of 128 K whose accumulators share one 128-column TMEM buffer before
// the epilogue drains it: each chunk adds two 64-K groups of np columns, so
// blocks of up to 16 tokens drain every 4 chunks, up to 32 every 2.
__host__ __device__ inline int unit_chunks(int np) { return np <= 16 ? 4 : np <= 32 ? 2 : 1; }
__host__ __device__ inline int blocks_of(int cnt) { return (cnt + kBlkTokens - 1) / kBlkTokens; }
__host__ __device__ inline int rows_of(int cnt) {  // packed rows of an entry with cnt tokens
  return (cnt / kBlkTokens) * kBlkTokens + round16(cnt % kBlkTokens);
}

bool prefill_tc_ok(const LayerArgs& a, int T) {
  return T >= kPrefillTcMin && T <= kMaxTokens && a.H % 128 == 0 && a.F % 128 == 0 && a.Fs % 128 == 0;
}

// ---------------------------------------------------------------------------
// scratch layout
// ---------------------------------------------------------------------------
struct PfLayout {
  size_t hdr, blk, xc, sx, hc_hi, hc_lo, sh, y_pair, y_sh, inv, total;
  int rows_cap, blk_cap;
};

static PfLayout pf_layout(const LayerArgs& a, int T) {
  PfLayout L{};
  const size_t H = a.H, k = a.k, Fm = std::max(a.F, a.Fs);
  const int pairs = T * a.k, has_sh = a.Fs > 0;
  const int nact = std::min(a.E, pairs);
  L.rows_cap = (has_sh ? rows_of(T) : 0) + pairs + 15 * nact;
  L.blk_cap = (has_sh ? blocks_of(T) : 0) + nact + pairs / kBlkTokens + 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  const size_t rows = L.rows_cap;
  L.hdr = take(256);
  L.blk = take(static_cast<size_t>(L.blk_cap) * sizeof(PBlk));
  L.xc = take(rows * H * 2);
  L.sx = take(rows * (H / 64) * 4);
  L.hc_hi = take(rows * Fm * 2);
  L.hc_lo = take(rows * Fm * 2);
  L.sh = take(rows * (Fm / 64) * 4);
  L.y_pair = take(static_cast<size_t>(pairs) * H * 4);
  L.y_sh = take(has_sh ? static_cast<size_t>(T) * H * 4 : 0);
  L.inv = take(static_cast<size_t>(pairs) * 4);
  (void)k;
  L.total = off;
  return L;
}

size_t prefill_workspace_bytes(const LayerArgs& a, int T) {
  return prefill_tc_ok(a, T) ? pf_layout(a, T).total : 0;
}

// ---------------------------------------------------------------------------
// pack: block table, activations in core-matrix order, group sums
// ---------------------------------------------------------------------------
constexpr int kPackThreads = 256;
constexpr int kPackSlices = kMaxTokens / 16;  // CTAs per entry: 16 packed rows each

__device__ __forceinline__ int clamp_nact(const LayerArgs& a) {
  const int n = *reinterpret_cast<volatile int*>(a.ws.n_act);
  return n < 0 ? 0 : (n > a.E ? a.E : n);
}

__device__ __forceinline__ int entry_cnt(const LayerArgs& a, int i, int has_sh) {
  if (has_sh && i == 0) return a.T;
  const int c = a.ws.act_cnt[i - has_sh];
  return c < 0 ? 0 : (c > a.T ? a.T : c);
}

__global__ void __launch_bounds__(kPackThreads) pf_pack_kernel(const __grid_constant__ LayerArgs a) {
  const int has_sh = a.Fs > 0 ? 1 : 0;
  const int n_ent = has_sh + clamp_nact(a);
  const int j = blockIdx.x / kPackSlices, slice = blockIdx.x % kPackSlices;  // entry, row slice
  if (j >= n_ent) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, H = a.H;
  const bool shared = has_sh && j == 0;
  const int Fj = shared ? a.Fs : a.F;
  const int cnt = entry_cnt(a, j, has_sh);
  // slices past the entry's packed rows have nothing to do (slice 0 also
  // writes the block table and the pair index)
  if (slice > 0 && slice * 16 >= rows_of(cnt)) return;

  // prefix over the entries before j: blocks, packed rows, packed h elements
  __shared__ long long s_red[3][kPackThreads / 32];
  long long nb = 0, rows = 0, helem = 0;
  for (int i = tid; i < j; i += kPackThreads) {
    const int c = entry_cnt(a, i, has_sh);
    nb += blocks_of(c);
    rows += rows_of(c);
    helem += static_cast<long long>(rows_of(c)) * ((has_sh && i == 0) ? a.Fs : a.F);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    nb += __shfl_xor_sync(kAllLanes, nb, o);
    rows += __shfl_xor_sync(kAllLanes, rows, o);
    helem += __shfl_xor_sync(kAllLanes, helem, o);
  }
  if (lane == 0) s_red[0][warp] = nb, s_red[1][warp] = rows, s_red[2][warp] = helem;
  __syncthreads();
  long long nb0 = 0, row0 = 0, h0 = 0;
  for (int w = 0; w < kPackThreads / 32; ++w) nb0 += s_red[0][w], row0 += s_red[1][w], h0 += s_red[2][w];

  const int nbj = blocks_of(cnt);
  const int expert = shared ? -1 : a.ws.act_expert[j - has_sh];
  const int pair0 = shared ? 0 : a.ws.act_off[j - has_sh];
  if (slice == 0 && tid < nbj) {
    const int b = tid;
    PBlk p;
    p.expert = expert;
    p.len = min(kBlkTokens, cnt - b * kBlkTokens);
    p.np = round16(p.len);
    p.xrow = static_cast<int>(row0) + b * kBlkTokens;
    p.tok0 = pair0 + b * kBlkTokens;
    p.hoff = static_cast<int>(h0) + b * kBlkTokens * Fj;
    p.entry = j;
    p.pad = 0;
    a.pf.blk[nb0 + b] = p;
  }
  if (slice == 0 && j == n_ent - 1 && tid == 0) {
    a.pf.hdr[0] = static_cast<int>(nb0) + nbj;
    a.pf.hdr[1] = has_sh ? blocks_of(a.T) : 0;
  }
  if (!shared && slice == 0)
    for (int n = tid; n < cnt; n += kPackThreads) {
      const int p = pair0 + n;
      const int slot = a.ws.pair_slot[p];
      if (slot >= 0 && slot < a.T * a.k) a.pf.inv[slot] = p;
    }

  // packed rows: one warp per row (this CTA's slice of 16 rows); a lane
  // handles 8 consecutive K values
  const int nrows = min(rows_of(cnt), (slice + 1) * 16), units = H / 8;
  for (int n = slice * 16 + warp; n < nrows; n += kPackThreads / 32) {
    const int b = n / kBlkTokens, nn = n % kBlkTokens;
    const int len = min(kBlkTokens, cnt - b * kBlkTokens), np = round16(len);
    const int xrow = static_cast<int>(row0) + b * kBlkTokens;
    int tok = -1;
    if (nn < len) tok = shared ? b * kBlkTokens + nn : a.ws.pair_token[pair0 + b * kBlkTokens + nn];
    if (tok < 0 || tok >= a.T) tok = -1;
    uint16_t* xb = a.pf.xc + static_cast<size_t>(xrow) * H;
    float* sxb = a.pf.sx + static_cast<size_t>(xrow) * (H / 64);
    // batches of 8 units per lane: every load of a batch is in flight
    // before the first one is used
    constexpr int kBatch = 8;
    for (int u0 = 0; u0 < units; u0 += 32 * kBatch) {
      uint4 vb[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int u = u0 + q * 32 + lane;
        vb[q] = make_uint4(0, 0, 0, 0);
        if (u < units && tok >= 0) vb[q] = __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(tok) * H) + u);
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int u = u0 + q * 32 + lane;
        if (u0 + q * 32 >= units) break;  // the same on every lane
        const uint4 v = vb[q];
        float s = bf16lo(v.x) + bf16hi(v.x) + bf16lo(v.y) + bf16hi(v.y) + bf16lo(v.z) + bf16hi(v.z) +
                  bf16lo(v.w) + bf16hi(v.w);
        // group sum over the 8 lanes (64 values) of this lane's group
        s += __shfl_xor_sync(kAllLanes, s, 1);
        s += __shfl_xor_sync(kAllLanes, s, 2);
        s += __shfl_xor_sync(kAllLanes, s, 4);
        if (u < units) {
          // K order inside the core row: 0,4,1,5,2,6,3,7
          uint4 w;
          w.x = __byte_perm(v.x, v.z, 0x5410);
          w.y = __byte_perm(v.x, v.z, 0x7632);
          w.z = __byte_perm(v.y, v.w, 0x5410);
          w.w = __byte_perm(v.y, v.w, 0x7632);
          const int c = u >> 4, k8 = u & 15;
          const size_t e = static_cast<size_t>(c) * np * 128 + (k8 * (np >> 3) + (nn >> 3)) * 64 + (nn & 7) * 8;
          *reinterpret_cast<uint4*>(xb + e) = w;
          if ((lane & 7) == 0) sxb[(u >> 3) * np + nn] = s;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// grouped GEMM on the tensor cores
// ---------------------------------------------------------------------------
constexpr int kPgThreads = 384;  // 12 warps
constexpr int kEpiWarps = 4, kDqWarps = 4, kBWarp = 8, kProdWarp = 9, kMmaWarp = 10;
constexpr int kMmaWarps = 2;  // MMA issuers: warp kMmaWarp + i issues the chunks with index % 2 == i
constexpr int kDqWarp0 = kEpiWarps;  // dequantise warps: kDqWarp0 .. kDqWarp0 + kDqWarps - 1
static_assert(kEpiWarps == 4 && kDqWarps == 4, "one epilogue and one dequantising warp per TMEM lane quarter");
static_assert(kDqWarp0 + kDqWarps <= kBWarp && kBWarp < kProdWarp && kProdWarp < kMmaWarp &&
                  kMmaWarp + kMmaWarps == kPgThreads / 32,
              "warp roles must not overlap");
static_assert(kDqWarps * 32 == 128, "one dequantising thread per A row");
template <int MODE>
constexpr int kNSC = MODE == 0 ? 16 : 10;  // code stages (8 KB each)
template <int MODE>
constexpr int kNSB = 4;  // activation (B) stages
constexpr int kNSA = 4;                  // A stages (in TMEM)

constexpr int kCodesStage = 128 * 64;    // 128 rows x 64 B (128 codes)
constexpr int kACols = 64;               // TMEM columns of one A stage: 128 bf16 per row
constexpr int kTmemBufs = 2;             // accumulator buffers of 128 columns each
constexpr int kACol0 = kTmemBufs * 128;  // A stages follow the accumulators
constexpr int kTmemCols = 512;
static_assert(kACol0 + kNSA * kACols <= kTmemCols, "TMEM columns");
constexpr int kNSG = 16;                 // group-sum stages (2 groups x 64 floats)
constexpr int kXPitch = 65;              // floats per row of the SwiGLU exchange (no bank conflicts)

struct PgSmem {
  int codes, b, gs, xchg, bars, total, bstage;
};

__host__ __device__ inline PgSmem pg_smem(int mode) {
  PgSmem L;
  int off = 0;
  L.codes = off;
  off += (mode == 0 ? kNSC<0> : kNSC<1>) * kCodesStage;
  L.bstage = kBlkTokens * 256 * (mode == 1 ? 2 : 1);
  L.b = off;
  off += (mode == 0 ? kNSB<0> : kNSB<1>) * L.bstage;
  L.gs = off;
  off += kNSG * 2 * kBlkTokens * 4;
  L.xchg = off;
  off += mode == 0 ? 64 * kXPitch * 4 : 0;
  L.bars = off;
  off += 1024;  // mbarriers, the TMEM address and the abort flag
  L.total = off;
  return L;
}

struct PgItem {
  PBlk blk;
  int tile, K, nch;
  const uint8_t* rec;
  const RecordOffsets* off;
  int Fe;
};

template <int MODE>
__device__ __forceinline__ bool pg_item(const LayerArgs& a, int it, int nblk, int nsb, PgItem& I) {
  const int has_sh = a.Fs > 0 ? 1 : 0;
  int b, tile;
  if (MODE == 0) {
    const int Ts = a.Fs / 64, Tr = a.F / 64;
    if (it < nsb * Ts) b = it / Ts, tile = it % Ts;
    else b = nsb + (it - nsb * Ts) / Tr, tile = (it - nsb * Ts) % Tr;
  } else {
    const int Th = a.H / 128;
    b = it / Th, tile = it % Th;
  }
  if (b >= nblk) return false;
  I.blk = a.pf.blk[b];
  I.tile = tile;
  const bool shared = has_sh && I.blk.expert < 0;
  I.Fe = shared ? a.Fs : a.F;
  I.K = MODE == 0 ? a.H : I.Fe;
  I.nch = I.K / 128;
  if (shared) {
    I.rec = a.shared, I.off = &a.off_s;
  } else {
    int e = I.blk.expert;
    if (e < 0 || e >= a.E) e = 0;
    I.blk.expert = e;
    I.rec = a.records + static_cast<size_t>(e) * a.off_r.stride;
    I.off = &a.off_r;
  }
  int np = I.blk.np;
  I.blk.np = np < 16 ? 16 : (np > kBlkTokens ? kBlkTokens : np);
  return true;
}

// Order of a CTA's items.  The shared expert's items (the first S of the
// list) each cost several routed items: blocks of up to 64 tokens against
// about 16, and in the down GEMM K = Fs against F.  With S < G CTAs, CTA
// c < S takes shared item c first and then sits out the first K rounds of
// the routed items, which the other G - S CTAs share; every routed item is
// still taken exactly once.  An item's cost is modelled as its 128-K chunks
// x (tokens + 16), and K is the rounded cost ratio minus one.  Every role
// of a CTA walks the same sequence.
struct PgSched {
  int S, R, G, K;
};

template <int MODE>
__device__ __forceinline__ PgSched pg_sched_of(const LayerArgs& a, int nblk, int nsb) {
  PgSched p;
  p.G = static_cast<int>(gridDim.x);
  p.S = nsb * (MODE == 0 ? a.Fs / 64 : a.H / 128);
  p.R = (nblk - nsb) * (MODE == 0 ? a.F / 64 : a.H / 128);
  p.K = 0;
  if (p.S > 0 && p.S < p.G && p.R > 0) {
    const int np_s = min(kBlkTokens, round16(a.T));
    const int nch_s = (MODE == 0 ? a.H : a.Fs) / 128, nch_r = (MODE == 0 ? a.H : a.F) / 128;
    const int w = (nch_s * (np_s + 16) + nch_r * 16) / (nch_r * 32);
    p.K = max(0, min(w - 1, p.R / (p.G - p.S)));
  }
  return p;
}

// Item index of CTA c's j-th item, -1 past its last.
__device__ __forceinline__ int pg_next(const PgSched& p, int c, int j) {
  long long r;
  if (p.K == 0) {
    r = c + static_cast<long long>(j) * p.G;
    return r < p.S + p.R ? static_cast<int>(r) : -1;
  }
  if (c < p.S) {
    if (j == 0) return c;
    r = static_cast<long long>(p.K) * (p.G - p.S) + static_cast<long long>(j - 1) * p.G + c;
  } else if (j < p.K) {
    r = static_cast<long long>(j) * (p.G - p.S) + (c - p.S);
  } else {
    r = static_cast<long long>(p.K) * (p.G - p.S) + static_cast<long long>(j - p.K) * p.G + c;
  }
  return r < p.R ? p.S + static_cast<int>(r) : -1;
}

// Waits for a phase; gives up (and tells every other role through `abort`)
// after the bounded limit or when another role already gave up.
__device__ __forceinline__ bool pg_wait(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      latch_error(err, kErrTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool pg_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* err) {
  return __all_sync(kAllLanes, pg_wait(bar, parity, abort, err)) != 0;
}

// SiLU with the fast exponential and division (a few ulp, far inside the
// parity bound; the per-item SwiGLU of a whole tile is on the epilogue's
// critical path here).  silu(64) = 64 exactly, as the identity layer needs.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Asks L2 to fetch [p, p + bytes) (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// An item's weight rows are contiguous runs in the record (the code rows and
// their scale/bias rows); the tiled loads then read them from L2 instead of
// visiting each DRAM page once per 128-wide chunk.
template <int MODE>
__device__ __forceinline__ void prefetch_item(const PgItem& I, int H) {
  if (MODE == 0) {
    const size_t r0 = static_cast<size_t>(I.tile) * 64;
    const uint32_t cb = 64 * (H / 2), sb = 64 * (H / 16);
    prefetch_l2(I.rec + I.off->gate_codes + r0 * (H / 2), cb);
    prefetch_l2(I.rec + I.off->up_codes + r0 * (H / 2), cb);
    prefetch_l2(I.rec + I.off->gate_sb + r0 * (H / 16), sb);
    prefetch_l2(I.rec + I.off->up_sb + r0 * (H / 16), sb);
  } else {
    const size_t r0 = static_cast<size_t>(I.tile) * 128;
    prefetch_l2(I.rec + I.off->down_codes + r0 * (I.Fe / 2), 128 * (I.Fe / 2));
    prefetch_l2(I.rec + I.off->down_sb + r0 * (I.Fe / 16), 128 * (I.Fe / 16));
  }
}

// Two bf16 lanes holding 128 + q (bits 0x4300 | q) -> q, exactly:
// (128 + q) * 1 - 128 needs no rounding.
__device__ __forceinline__ uint32_t codes_bf16x2(uint32_t v) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(v), "r"(0x3F803F80u), "r"(0xC300C300u));
  return r;
}

// 12 warps put three warps on each SM sub-partition: 168 registers each.
template <int MODE>
__global__ void __maxnreg__(168)
    pf_gemm_kernel(const __grid_constant__ LayerArgs a, const __grid_constant__ PfMaps maps) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const PgSmem L = pg_smem(MODE);
  uint8_t* s_codes = smem + L.codes;
  uint8_t* s_b = smem + L.b;
  float* s_x = reinterpret_cast<float*>(smem + L.xchg);
  float* s_gs = reinterpret_cast<float*>(smem + L.gs);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* codes_full = bars;
  uint64_t* codes_empty = codes_full + kNSC<MODE>;
  uint64_t* a_full = codes_empty + kNSC<MODE>;
  uint64_t* a_empty = a_full + kNSA;
  uint64_t* b_full = a_empty + kNSA;
  uint64_t* b_empty = b_full + kNSB<MODE>;
  uint64_t* tm_full = b_empty + kNSB<MODE>;
  uint64_t* tm_empty = tm_full + kTmemBufs;
  uint64_t* gs_full = tm_empty + kTmemBufs;
  uint64_t* gs_empty = gs_full + kNSG;
  uint64_t* mma_done = gs_empty + kNSG;  // an issuer's own MMAs complete (abort path)
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(mma_done + kMmaWarps);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_taddr + 1);
  unsigned* err = &a.ws.ctl[0];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kNSC<MODE>; ++i) mbar_init(&codes_full[i], 1), mbar_init(&codes_empty[i], kDqWarps);
    for (int i = 0; i < kNSA; ++i) mbar_init(&a_full[i], kDqWarps), mbar_init(&a_empty[i], 1);
    for (int i = 0; i < kNSB<MODE>; ++i) mbar_init(&b_full[i], 1), mbar_init(&b_empty[i], 1);
    // tm_full: one commit from each MMA issuer per drain unit (an issuer
    // alone in a unit commits twice)
    for (int i = 0; i < kTmemBufs; ++i) mbar_init(&tm_full[i], kMmaWarps), mbar_init(&tm_empty[i], kEpiWarps);
    for (int i = 0; i < kMmaWarps; ++i) mbar_init(&mma_done[i], 1);
    for (int i = 0; i < kNSG; ++i) mbar_init(&gs_full[i], 1), mbar_init(&gs_empty[i], kEpiWarps);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) tmem_alloc(smem_u32(s_taddr), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = *s_taddr;

  int nblk = a.pf.hdr[0], nsb = a.pf.hdr[1];
  nblk = max(0, nblk);
  nsb = min(max(0, nsb), nblk);
  const int H = a.H;
  const PgSched ps = pg_sched_of<MODE>(a, nblk, nsb);
  const int cta = static_cast<int>(blockIdx.x);

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ codes
    const uint64_t pol = policy_evict_first();
    RingPos pc, pg;
    int issued = 0;
    bool stop = false;
    for (int j = 0, it; !stop && (it = pg_next(ps, cta, j)) >= 0; ++j) {
      PgItem I;
      if (!pg_item<MODE>(a, it, nblk, nsb, I)) break;
      if (lane == 0) {  // this item's rows (first item only) and the next item's, into L2
        PgItem J;
        if (j == 0) prefetch_item<MODE>(I, H);
        const int itn = pg_next(ps, cta, j + 1);
        if (itn >= 0 && pg_item<MODE>(a, itn, nblk, nsb, J)) prefetch_item<MODE>(J, H);
      }
      const int np = I.blk.np;
      const float* gsum = MODE == 0 ? a.pf.sx + static_cast<size_t>(I.blk.xrow) * (H / 64) : a.pf.sh + I.blk.hoff / 64;
      for (int c = 0; c < I.nch; ++c, pc.next(kNSC<MODE>), pg.next(kNSG)) {
        if (issued >= kNSC<MODE> && !pg_wait_warp(&codes_empty[pc.s], pc.ph ^ 1u, s_abort, err)) {
          stop = true;
          break;
        }
        if (issued >= kNSG && !pg_wait_warp(&gs_empty[pg.s], pg.ph ^ 1u, s_abort, err)) {
          stop = true;
          break;
        }
        if (lane == 0) {  // this chunk's two group sums of the block's tokens
          mbar_arrive_expect_tx(&gs_full[pg.s], 2 * np * 4);
          bulk_g2s(s_gs + pg.s * 2 * kBlkTokens, gsum + static_cast<size_t>(2 * c) * np, 2 * np * 4, &gs_full[pg.s]);
        }
        if (lane == 0) {  // the chunk's 128 rows x 64 B of codes: one or two tiled loads
          uint8_t* dst = s_codes + pc.s * kCodesStage;
          const bool sh = I.rec == a.shared;
          const CUtensorMap* m = sh ? maps.shared : maps.routed;
          const int z = sh ? 0 : I.blk.expert;
          mbar_arrive_expect_tx(&codes_full[pc.s], kCodesStage);
          if (MODE == 0) {
            tma_load_3d(dst, &m[0], c * 64, I.tile * 64, z, &codes_full[pc.s], pol);
            tma_load_3d(dst + 64 * 64, &m[1], c * 64, I.tile * 64, z, &codes_full[pc.s], pol);
          } else {
            tma_load_3d(dst, &m[0], c * 64, I.tile * 128, z, &codes_full[pc.s], pol);
          }
        }
        __syncwarp();
        ++issued;
      }
    }
    // copies in flight land before the CTA leaves
    for (int j = max(0, issued - kNSC<MODE>); j < issued; ++j)
      if (!mbar_wait(&codes_full[j % kNSC<MODE>], (j / kNSC<MODE>) & 1)) latch_error(err, kErrTimeout);
    for (int j = max(0, issued - kNSG); j < issued; ++j)
      if (!mbar_wait(&gs_full[j % kNSG], (j / kNSG) & 1)) latch_error(err, kErrTimeout);
  } else if (warp >= kDqWarp0 && warp < kDqWarp0 + kDqWarps) {
    // ------------------------------------------------------------ dequantise
    const int dw = warp - kDqWarp0, t = dw * 32 + lane;
    RingPos pc, pa;
    int cc = 0;
    for (int j = 0, it; !*s_abort && (it = pg_next(ps, cta, j)) >= 0; ++j) {
      PgItem I;
      if (!pg_item<MODE>(a, it, nblk, nsb, I)) break;
      bool stop = false;
      for (int c = 0; c < I.nch; ++c, ++cc, pc.next(kNSC<MODE>), pa.next(kNSA)) {
        if (cc >= kNSA && !pg_wait_warp(&a_empty[pa.s], pa.ph ^ 1u, s_abort, err)) {
          stop = true;
          break;
        }
        if (!pg_wait_warp(&codes_full[pc.s], pc.ph, s_abort, err)) {
          stop = true;
          break;
        }
        // One row per thread: row = TMEM lane.  The code tile lands with the
        // 64-byte swizzle (16-byte chunk j of row r at chunk j ^ ((r >> 1) & 3)),
        // so 8 consecutive rows reading the same logical chunk hit distinct
        // banks.  Word k8 of the row (8 codes) becomes TMEM columns 4k8..4k8+3.
        tc_fence_after();
        const uint8_t* src = s_codes + pc.s * kCodesStage + t * 64;
        const int sw = (t >> 1) & 3;
        const uint32_t ta = taddr + (static_cast<uint32_t>(dw * 32) << 16) + kACol0 + pa.s * kACols;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 q = *reinterpret_cast<const uint4*>(src + ((j ^ sw) << 4));
          const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
          uint32_t v[16];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t x = w4[w];
            v[4 * w + 0] = codes_bf16x2((x & 0x000F000Fu) | 0x43004300u);
            v[4 * w + 1] = codes_bf16x2(((x >> 4) & 0x000F000Fu) | 0x43004300u);
            v[4 * w + 2] = codes_bf16x2(((x >> 8) & 0x000F000Fu) | 0x43004300u);
            v[4 * w + 3] = codes_bf16x2(((x >> 12) & 0x000F000Fu) | 0x43004300u);
          }
          tmem_st16(ta + j * 16, v);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&a_full[pa.s]);
          mbar_arrive(&codes_empty[pc.s]);
        }
      }
      if (stop) break;
    }
  } else if (warp == kBWarp) {
    // ------------------------------------------------------------ B operand
    if (lane == 0) {
      RingPos pb;
      int issued = 0;
      bool stop = false;
      for (int j = 0, it; !stop && (it = pg_next(ps, cta, j)) >= 0; ++j) {
        PgItem I;
        if (!pg_item<MODE>(a, it, nblk, nsb, I)) break;
        const int np = I.blk.np;
        for (int c = 0; c < I.nch; ++c, pb.next(kNSB<MODE>)) {
          if (issued >= kNSB<MODE> && !pg_wait(&b_empty[pb.s], pb.ph ^ 1u, s_abort, err)) {
            stop = true;
            break;
          }
          uint8_t* bdst = s_b + pb.s * L.bstage;
          const uint32_t part = np * 256;
          if (MODE == 0) {
            mbar_arrive_expect_tx(&b_full[pb.s], part);
            bulk_g2s(bdst, a.pf.xc + static_cast<size_t>(I.blk.xrow) * H + static_cast<size_t>(c) * np * 128, part,
                     &b_full[pb.s]);
          } else {
            const size_t e = static_cast<size_t>(I.blk.hoff) + static_cast<size_t>(c) * np * 128;
            mbar_arrive_expect_tx(&b_full[pb.s], 2 * part);
            bulk_g2s(bdst, a.pf.hc_hi + e, part, &b_full[pb.s]);
            bulk_g2s(bdst + part, a.pf.hc_lo + e, part, &b_full[pb.s]);
          }
          ++issued;
        }
      }
      for (int j = max(0, issued - kNSB<MODE>); j < issued; ++j)
        if (!mbar_wait(&b_full[j % kNSB<MODE>], (j / kNSB<MODE>) & 1)) latch_error(err, kErrTimeout);
    }
    __syncwarp();
  } else if (warp >= kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // Two issuing threads: one thread can issue a tcgen05.mma only every
    // ~50 cycles, two together about every 30.  Issuer mi takes the chunks
    // with index % 2 == mi; both track every ring.  The accumulators of the
    // chunks of one drain unit share a TMEM buffer: chunk j of the unit puts
    // its groups at columns (2j + gi) * np.
    const int mi = warp - kMmaWarp;
    if (lane == 0) {
      RingPos pa, pb;
      int cc = 0, units = 0;
      bool stop = false;
      for (int j = 0, it; !stop && (it = pg_next(ps, cta, j)) >= 0; ++j) {
        PgItem I;
        if (!pg_item<MODE>(a, it, nblk, nsb, I)) break;
        const int np = I.blk.np, U = unit_chunks(np);
        const uint32_t idesc = idesc_bf16_f32(128, np);
        for (int u0 = 0; u0 < I.nch && !stop; u0 += U, ++units) {
          const int ue = min(u0 + U, I.nch), buf = units % kTmemBufs;
          const uint32_t uph = (units / kTmemBufs) & 1;
          int mine = 0, others = 0;
          for (int c = u0; c < ue; ++c, ++cc, pa.next(kNSA), pb.next(kNSB<MODE>)) {
            if ((cc % kMmaWarps) != mi) {
              ++others;
              continue;
            }
            if ((mine == 0 && units >= kTmemBufs && !pg_wait(&tm_empty[buf], uph ^ 1u, s_abort, err)) ||
                !pg_wait(&a_full[pa.s], pa.ph, s_abort, err) || !pg_wait(&b_full[pb.s], pb.ph, s_abort, err)) {
              stop = true;
              break;
            }
            ++mine;
            tc_fence_after();
            const uint32_t a0 = taddr + kACol0 + pa.s * kACols, b0 = smem_u32(s_b + pb.s * L.bstage);
            // descriptor of the chunk's first K step; each next step adds
            // np * 32 bytes to the start address field (units of 16 bytes)
            const uint64_t bd0 = smem_desc(b0, np * 16, 128), bstep = static_cast<uint64_t>(np * 2);
            const uint64_t bd_lo = smem_desc(b0 + np * 256, np * 16, 128);
#pragma unroll
            for (int gi = 0; gi < 2; ++gi) {
              const uint32_t d = taddr + buf * 128 + (2 * (c - u0) + gi) * np;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const int kq = gi * 4 + kk;  // K = 16 per MMA: 8 TMEM columns of A
                mma_bf16_ta(d, a0 + kq * 8, bd0 + kq * bstep, idesc, kk > 0 ? 1u : 0u);
                if (MODE == 1) mma_bf16_ta(d, a0 + kq * 8, bd_lo + kq * bstep, idesc, 1u);
              }
            }
            mma_commit(smem_u32(&a_empty[pa.s]));
            mma_commit(smem_u32(&b_empty[pb.s]));
          }
          if (stop) break;
          if (mine > 0) {
            mma_commit(smem_u32(&tm_full[buf]));
            if (others == 0) mma_commit(smem_u32(&tm_full[buf]));
          }
        }
      }
      // Normally the epilogue has consumed every accumulator (so every MMA
      // completed) before the final barrier; after an abort, this issuer's
      // MMAs land before TMEM is released.
      if (*s_abort) {
        mma_commit(smem_u32(&mma_done[mi]));
        if (!mbar_wait(&mma_done[mi], 0)) latch_error(err, kErrTimeout);
      }
    }
    __syncwarp();
  } else if (warp < kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int q = warp;              // TMEM lane quarter
    const int row = q * 32 + lane;   // TMEM lane = A row of the item
    RingPos pg;
    int units = 0;
    bool stop = false;
    for (int j = 0, it; !stop && (it = pg_next(ps, cta, j)) >= 0; ++j) {
      PgItem I;
      if (!pg_item<MODE>(a, it, nblk, nsb, I)) break;
      const int np = I.blk.np, U = unit_chunks(np);
      const int G = I.K / 64;
      // this row's scale/bias words (the next chunk's pair is loaded one chunk ahead)
      const uint32_t* sbrow;
      if (MODE == 0) {
        const uint64_t o = row < 64 ? I.off->gate_sb : I.off->up_sb;
        sbrow = reinterpret_cast<const uint32_t*>(I.rec + o) + static_cast<size_t>(I.tile * 64 + (row & 63)) * G;
      } else {
        sbrow = reinterpret_cast<const uint32_t*>(I.rec + I.off->down_sb) + static_cast<size_t>(I.tile * 128 + row) * G;
      }
      float acc[kBlkTokens];
#pragma unroll
      for (int j = 0; j < kBlkTokens; ++j) acc[j] = 0.f;
      // the row's scale/bias words of the next four chunks are in flight
      // while a chunk is drained (an L2 round trip takes longer than one
      // chunk's epilogue)
      const uint2* sbp = reinterpret_cast<const uint2*>(sbrow);
      uint2 sb0 = __ldg(sbp), sb1 = make_uint2(0, 0), sb2 = make_uint2(0, 0), sb3 = make_uint2(0, 0);
      if (1 < I.nch) sb1 = __ldg(sbp + 1);
      if (2 < I.nch) sb2 = __ldg(sbp + 2);
      if (3 < I.nch) sb3 = __ldg(sbp + 3);
      for (int u0 = 0; u0 < I.nch && !stop; u0 += U, ++units) {
        const int ue = min(u0 + U, I.nch), buf = units % kTmemBufs;
        const uint32_t uph = (units / kTmemBufs) & 1;
        // the epilogue warps decide together, so the barriers below stay uniform
        if (named_bar_or(2, kEpiWarps * 32, !pg_wait_warp(&tm_full[buf], uph, s_abort, err))) {
          stop = true;
          break;
        }
        // A failed wait inside the unit only marks the warp; the four
        // epilogue warps agree at the unit's end, so no named barrier runs
        // per chunk and the barriers after it stay uniform.
        bool lost = false;
        for (int c = u0; c < ue; ++c, pg.next(kNSG)) {
          const uint32_t sbw[2] = {sb0.x, sb0.y};
          sb0 = sb1, sb1 = sb2, sb2 = sb3;
          if (c + 4 < I.nch) sb3 = __ldg(sbp + c + 4);
          if (!lost && !pg_wait_warp(&gs_full[pg.s], pg.ph, s_abort, err)) lost = true;
          tc_fence_after();
          const uint32_t base0 =
              taddr + (static_cast<uint32_t>(q * 32) << 16) + buf * 128 + (2 * (c - u0)) * np;
          const uint32_t base1 = base0 + np;
          const float s0 = bf16lo(sbw[0]), b0 = bf16hi(sbw[0]), s1 = bf16lo(sbw[1]), b1 = bf16hi(sbw[1]);
          const float* gs0 = s_gs + pg.s * 2 * kBlkTokens;
          const float* gs1 = gs0 + np;
#pragma unroll
          for (int p = 0; p < kBlkTokens / 16; ++p)  // 16 columns of both groups per TMEM round trip
            if (p * 16 < np) {
              uint32_t d0[8], d1[8], e0[8], e1[8];
              tmem_ld8(base0 + p * 16, d0);
              tmem_ld8(base0 + p * 16 + 8, d1);
              tmem_ld8(base1 + p * 16, e0);
              tmem_ld8(base1 + p * 16 + 8, e1);
              float xa[16], xb[16];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float4 ua = *reinterpret_cast<const float4*>(gs0 + p * 16 + 4 * j);
                const float4 ub = *reinterpret_cast<const float4*>(gs1 + p * 16 + 4 * j);
                xa[4 * j] = ua.x, xa[4 * j + 1] = ua.y, xa[4 * j + 2] = ua.z, xa[4 * j + 3] = ua.w;
                xb[4 * j] = ub.x, xb[4 * j + 1] = ub.y, xb[4 * j + 2] = ub.z, xb[4 * j + 3] = ub.w;
              }
              tmem_wait();
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                float v = fmaf(s0, __uint_as_float(d0[j]), fmaf(b0, xa[j], acc[p * 16 + j]));
                acc[p * 16 + j] = fmaf(s1, __uint_as_float(e0[j]), fmaf(b1, xb[j], v));
                float w = fmaf(s0, __uint_as_float(d1[j]), fmaf(b0, xa[8 + j], acc[p * 16 + 8 + j]));
                acc[p * 16 + 8 + j] = fmaf(s1, __uint_as_float(e1[j]), fmaf(b1, xb[8 + j], w));
              }
            }
          __syncwarp();
          if (lane == 0) mbar_arrive(&gs_empty[pg.s]);
        }
        if (named_bar_or(2, kEpiWarps * 32, lost)) stop = true;
        if (stop) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tm_empty[buf]);
      }
      if (stop) break;
      if (MODE == 0) {
        // SwiGLU: up rows (64..127, warps 2-3) hand their values to the gate rows
        // (np is a multiple of 16: one test per 16 tokens, so each block of
        // 16 is straight-line code whose exponentials and divisions overlap)
        if (q >= 2) {
          float* xr = s_x + ((q - 2) * 32 + lane) * kXPitch;
#pragma unroll
          for (int j0 = 0; j0 < kBlkTokens; j0 += 16)
            if (j0 < np)
#pragma unroll
              for (int j = j0; j < j0 + 16; ++j) xr[j] = acc[j];
        }
        named_bar(1, kEpiWarps * 32);
        if (q < 2) {  // h = silu(g) * u of the tile's 64 rows, into the exchange rows
          float* xr = s_x + row * kXPitch;
#pragma unroll
          for (int n0 = 0; n0 < kBlkTokens; n0 += 16)
            if (n0 < np) {
              float u[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) u[j] = xr[n0 + j];
#pragma unroll
              for (int j = 0; j < 16; ++j) xr[n0 + j] = silu_f(acc[n0 + j]) * u[j];
            }
        }
        named_bar(1, kEpiWarps * 32);
        // The tile's h in the down GEMM's B layout (bf16 hi + lo): its 64
        // rows are 8 k8 columns of one 128-K chunk, a contiguous run of
        // 8 * np 16-byte core rows: core row (k8l, token n) holds rows
        // 8 k8l + {0, 4, 1, 5, 2, 6, 3, 7} of token n.  Each thread builds
        // whole core rows from the exchange and stores them as 16 bytes.
        {
          const int cf = I.tile >> 1, k80 = 8 * (I.tile & 1), r8n = np >> 3;
          const size_t base = static_cast<size_t>(I.blk.hoff) + static_cast<size_t>(cf) * np * 128 +
                              static_cast<size_t>(k80) * r8n * 64;
          for (int u = tid; u < 8 * np; u += kEpiWarps * 32) {
            const int k8l = u / np, n = u - k8l * np;
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float h0 = s_x[(8 * k8l + j) * kXPitch + n], h1 = s_x[(8 * k8l + 4 + j) * kXPitch + n];
              const uint16_t a0 = f32_to_bf16_rne(h0), a1 = f32_to_bf16_rne(h1);
              const uint16_t b0 = f32_to_bf16_rne(h0 - __uint_as_float(static_cast<uint32_t>(a0) << 16));
              const uint16_t b1 = f32_to_bf16_rne(h1 - __uint_as_float(static_cast<uint32_t>(a1) << 16));
              hw[j] = static_cast<uint32_t>(a0) | (static_cast<uint32_t>(a1) << 16);
              lw[j] = static_cast<uint32_t>(b0) | (static_cast<uint32_t>(b1) << 16);
            }
            // core row (k8l, r8 = n / 8, n % 8) at element (k8l * r8n + n / 8) * 64 + (n % 8) * 8
            const size_t e = base + (static_cast<size_t>(k8l) * r8n + (n >> 3)) * 64 + (n & 7) * 8;
            *reinterpret_cast<uint4*>(a.pf.hc_hi + e) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(a.pf.hc_lo + e) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        // group sums of h over the tile's 64 rows (one group of the down
        // GEMM): eight threads per token, each over 8 rows, then a fixed
        // butterfly (the same order every time)
        {
          const int n = tid >> 3, part = tid & 7;
          float sum = 0.f;
          if (n < np)
#pragma unroll
            for (int r = 0; r < 8; ++r) sum += s_x[(8 * part + r) * kXPitch + n];
          sum += __shfl_xor_sync(kAllLanes, sum, 1);
          sum += __shfl_xor_sync(kAllLanes, sum, 2);
          sum += __shfl_xor_sync(kAllLanes, sum, 4);
          if (n < np && part == 0) a.pf.sh[I.blk.hoff / 64 + I.tile * np + n] = sum;
          if (np > 16) {  // tokens 16 .. np - 1: a second round
            const int n2 = n + 16;
            float s2 = 0.f;
            if (n2 < np)
#pragma unroll
              for (int r = 0; r < 8; ++r) s2 += s_x[(8 * part + r) * kXPitch + n2];
            s2 += __shfl_xor_sync(kAllLanes, s2, 1);
            s2 += __shfl_xor_sync(kAllLanes, s2, 2);
            s2 += __shfl_xor_sync(kAllLanes, s2, 4);
            if (n2 < np && part == 0) a.pf.sh[I.blk.hoff / 64 + I.tile * np + n2] = s2;
            if (np > 32) {
#pragma unroll
              for (int rr = 2; rr < 4; ++rr) {
                const int n3 = n + 16 * rr;
                float s3 = 0.f;
                if (n3 < np)
#pragma unroll
                  for (int r = 0; r < 8; ++r) s3 += s_x[(8 * part + r) * kXPitch + n3];
                s3 += __shfl_xor_sync(kAllLanes, s3, 1);
                s3 += __shfl_xor_sync(kAllLanes, s3, 2);
                s3 += __shfl_xor_sync(kAllLanes, s3, 4);
                if (n3 < np && part == 0) a.pf.sh[I.blk.hoff / 64 + I.tile * np + n3] = s3;
              }
            }
          }
        }
        named_bar(1, kEpiWarps * 32);
      } else {
        const int r = I.tile * 128 + row;
        const bool shared = a.Fs > 0 && I.blk.expert < 0;
        float* y = shared ? a.pf.y_sh : a.pf.y_pair;
#pragma unroll
        for (int n = 0; n < kBlkTokens; ++n)
          if (n < I.blk.len) y[static_cast<size_t>(I.blk.tok0 + n) * H + r] = acc[n];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(taddr, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// combine: out = y_shared + sum_i p_i y_{e_i}
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) pf_combine_kernel(const __grid_constant__ LayerArgs a) {
  const int t = blockIdx.x, H = a.H, k = a.k;
  const bool has_sh = a.Fs > 0;
  // the token's pair rows and weights, read once into shared memory
  __shared__ int s_p[kMaxTopK];
  __shared__ float s_w[kMaxTopK];
  if (threadIdx.x < k) {
    int p = a.pf.inv[t * k + threadIdx.x];
    if (p < 0 || p >= a.T * k) p = 0;
    s_p[threadIdx.x] = p;
    s_w[threadIdx.x] = a.weights[t * k + threadIdx.x];
  }
  __syncthreads();
  for (int r4 = threadIdx.x; r4 < H / 4; r4 += blockDim.x) {
    float4 acc = has_sh ? reinterpret_cast<const float4*>(a.pf.y_sh + static_cast<size_t>(t) * H)[r4]
                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int i = 0; i < k; ++i) {
      const float w = s_w[i];
      const float4 y = reinterpret_cast<const float4*>(a.pf.y_pair + static_cast<size_t>(s_p[i]) * H)[r4];
      acc.x = fmaf(w, y.x, acc.x), acc.y = fmaf(w, y.y, acc.y);
      acc.z = fmaf(w, y.z, acc.z), acc.w = fmaf(w, y.w, acc.w);
    }
    const size_t o = static_cast<size_t>(t) * H + r4 * 4;
    if (a.out_f32) *reinterpret_cast<float4*>(a.out_f32 + o) = acc;
    uint2 b;
    b.x = static_cast<uint32_t>(f32_to_bf16_rne(acc.x)) | (static_cast<uint32_t>(f32_to_bf16_rne(acc.y)) << 16);
    b.y = static_cast<uint32_t>(f32_to_bf16_rne(acc.z)) | (static_cast<uint32_t>(f32_to_bf16_rne(acc.w)) << 16);
    *reinterpret_cast<uint2*>(a.out_bf16 + o) = b;
  }
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------
size_t prefill_smem_need(const LayerArgs&, int) { return std::max(pg_smem(0).total, pg_smem(1).total); }

cudaError_t set_prefill_attributes(int smem_optin) {
  const void* fns[] = {(const void*)pf_gemm_kernel<0>, (const void*)pf_gemm_kernel<1>};
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

static cudaError_t markp(const LayerArgs& a, int i, cudaStream_t st) {
  return a.prof_on ? cudaEventRecord(static_cast<cudaEvent_t>(a.prof[i]), st) : cudaSuccess;
}

// Tensor maps of a layer's code matrices (routed records and the shared
// record) for the tiled loads of the prefill kernels.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static bool encode_codes(EncodeTiledFn enc, CUtensorMap* m, const uint8_t* base, uint64_t row_bytes, uint64_t rows,
                         uint64_t n_rec, uint64_t rec_stride, uint32_t box_rows) {
  const cuuint64_t dim[3] = {row_bytes, rows, n_rec};
  const cuuint64_t stride[2] = {row_bytes, rec_stride};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(base), dim, stride, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Fills `out` (valid = 1) when the layer can take the tensor-core prefill
// path; valid = 0 otherwise (no records, or shapes the path does not take).
cudaError_t build_layer_maps(const LayerArgs& a, LayerMaps* out) {
  out->valid = 0;
  if (!a.records || a.H % 128 || a.F % 128 || a.Fs % 128) return cudaSuccess;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return e ? e : cudaErrorNotSupported;
  EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(fn);
  const uint64_t H = a.H, F = a.F, Fs = a.Fs, E = a.E;
  bool ok = encode_codes(enc, &out->gateup.routed[0], a.records + a.off_r.gate_codes, H / 2, F, E, a.off_r.stride, 64) &&
            encode_codes(enc, &out->gateup.routed[1], a.records + a.off_r.up_codes, H / 2, F, E, a.off_r.stride, 64) &&
            encode_codes(enc, &out->down.routed[0], a.records + a.off_r.down_codes, F / 2, H, E, a.off_r.stride, 128);
  out->down.routed[1] = out->down.routed[0];
  if (ok && a.shared) {
    ok = encode_codes(enc, &out->gateup.shared[0], a.shared + a.off_s.gate_codes, H / 2, Fs, 1, a.off_s.stride, 64) &&
         encode_codes(enc, &out->gateup.shared[1], a.shared + a.off_s.up_codes, H / 2, Fs, 1, a.off_s.stride, 64) &&
         encode_codes(enc, &out->down.shared[0], a.shared + a.off_s.down_codes, Fs / 2, H, 1, a.off_s.stride, 128);
    out->down.shared[1] = out->down.shared[0];
  } else if (ok) {
    out->gateup.shared[0] = out->gateup.shared[1] = out->gateup.routed[0];
    out->down.shared[0] = out->down.shared[1] = out->down.routed[0];
  }
  if (!ok) return cudaErrorInvalidValue;
  out->valid = 1;
  return cudaSuccess;
}

cudaError_t launch_prefill(const LayerArgs& in, const LayerMaps* maps, int num_sms, cudaStream_t st) {
  if (!prefill_tc_ok(in, in.T) || !in.ws.pf || !maps || !maps->valid) return launch_decode(in, num_sms, st);
  LayerArgs a = in;
  const PfLayout L = pf_layout(a, a.T);
  uint8_t* base = a.ws.pf;
  a.pf.hdr = reinterpret_cast<int*>(base + L.hdr);
  a.pf.blk = reinterpret_cast<PBlk*>(base + L.blk);
  a.pf.xc = reinterpret_cast<uint16_t*>(base + L.xc);
  a.pf.sx = reinterpret_cast<float*>(base + L.sx);
  a.pf.hc_hi = reinterpret_cast<uint16_t*>(base + L.hc_hi);
  a.pf.hc_lo = reinterpret_cast<uint16_t*>(base + L.hc_lo);
  a.pf.sh = reinterpret_cast<float*>(base + L.sh);
  a.pf.y_pair = reinterpret_cast<float*>(base + L.y_pair);
  a.pf.y_sh = reinterpret_cast<float*>(base + L.y_sh);
  a.pf.inv = reinterpret_cast<int*>(base + L.inv);
  cudaError_t e;
  if ((e = markp(a, 0, st))) return e;
  if ((e = launch_decode_router(a, num_sms, st))) return e;
  pf_pack_kernel<<<(a.E + (a.Fs > 0 ? 1 : 0)) * kPackSlices, kPackThreads, 0, st>>>(a);
  if ((e = cudaGetLastError())) return e;
  if ((e = markp(a, 1, st))) return e;
  pf_gemm_kernel<0><<<num_sms, kPgThreads, pg_smem(0).total, st>>>(a, maps->gateup);
  if ((e = cudaGetLastError())) return e;
  if ((e = markp(a, 2, st))) return e;
  pf_gemm_kernel<1><<<num_sms, kPgThreads, pg_smem(1).total, st>>>(a, maps->down);
  if ((e = cudaGetLastError())) return e;
  pf_combine_kernel<<<a.T, 256, 0, st>>>(a);
  if ((e = cudaGetLastError())) return e;
  return markp(a, 3, st);
}

}  // namespace moe
