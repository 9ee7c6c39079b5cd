// kernels.h -- argument blocks shared by the host orchestration (api.cu) and
// the kernels (decode.cu, prefill.cu).  Host+device, no CUDA-only types in
// the structs themselves.
#pragma once

#include <cstddef>
#include <cstdint>

namespace moe {

constexpr int kMaxTokens = 128;  // decode B and prefill T cap
constexpr int kMaxTopK = 32;
constexpr int kMaxExperts = 1024;
constexpr int kMaxDim = 8192;    // H, F, Fs
constexpr int kBtMaxTokens = 16; // largest batch of the few-token fused path (decode_bt.cu)
constexpr int kConsumers = 256;  // consumer threads of the GEMV kernels (8 warps)
constexpr int kStages = 4;       // bulk-copy pipeline depth
constexpr int kStageTarget = 36 * 1024;  // bytes of weights per pipeline stage

// Error bits latched in the workspace control block by device code.
enum : unsigned {
  kErrTimeout = 1u,    // a bounded wait expired
  kErrResidency = 2u,  // a slot tag did not name the routed expert
  kErrRange = 4u,      // a routed id or count was out of range (clamped)
};

// Region offsets inside one expert record (see include/moe.h).
struct RecordOffsets {
  uint64_t gate_codes, up_codes, down_codes, gate_sb, up_sb, down_sb, bytes, stride;
};

// Device pointers into the caller's workspace (computed on the host).
struct Workspace {
  unsigned* ctl;         // [0] error bits, [1] router done counter, [2] gate|up (or fused
                         // kernel) item claims, [3] shared-only gate|up claims, [8] fused
                         // kernel producers done claiming, [10] router CTAs done writing xq
  unsigned* hcnt;        // fused kernels: gate|up items done per expert entry [kMaxExperts + 1]
  unsigned* tcnt;        // single token, fused kernel: experts done per down row tile
  uint8_t* hx;           // single token: fixed-point h, one block of 96 * nc bytes per
                         // expert entry (nc chunks, starting at byte 96 * c0): [4 kinds]
                         // [nc] uint4 words (word i of a uint4 = 8-value group i of the
                         // chunk), then [nc] float4 group 2^e, then [nc] float4 group sums
  float* ypart;          // fused kernels: [entry][H] (one token) or [pair][H] (few tokens)
                         // weighted down outputs
  uint8_t* xq;           // few-token fused path: the tokens' fixed-point activation chunks,
                         // [T][4 kinds][H/32] uint4 words, then [T][H/32] float2 (2^e, sum)
  float* logits;         // [T][E]
  int* n_act;            // number of distinct routed experts this step
  int* act_expert;       // [E] active expert ids, ascending
  int* act_off;          // [E] first pair of each active expert
  int* act_cnt;          // [E] tokens of each active expert
  int* pair_token;       // [T*k] token of each (expert, token) pair, grouped by expert
  int* pair_slot;        // [T*k] t*k + i position of the pair in ids/weights
  float* h;              // [T*k][F]  SwiGLU activations of routed pairs
  float* h_shared;       // [T][Fs]   SwiGLU activations of the shared expert
  uint16_t* x_stage;     // host-entry staging: [T][H] bf16
  uint16_t* ob_stage;    // [T][H] bf16
  float* of_stage;       // [T][H] f32
  int32_t* ids_stage;    // [T][k]
  float* w_stage;        // [T][k]
  uint8_t* pf;           // prefill chunk scratch (tensor-core path), or null
  float* rvq_g;          // residual-VQ layers, one token at a time: gate partial sums
                         // [input slice][entry][max(F, Fs)]
  float* rvq_u;          // up partial sums, same layout
  float* rvq_y;          // down partial sums [entry][input slice of F][H]
};

// One token block of the prefill path: up to 64 tokens of one expert (or of
// the shared expert), padded to a multiple of 16 rows.
struct PBlk {
  int expert;  // routed expert id, -1 for the shared expert
  int len;     // tokens in the block
  int np;      // len rounded up to a multiple of 16
  int xrow;    // first packed row of the block (activation blocks, group sums)
  int tok0;    // first pair position (routed) or first token (shared)
  int hoff;    // first element of the block's packed h (hi and lo arrays)
  int entry;   // 0.. (shared expert first, then active experts ascending)
  int pad;
};

// Prefill scratch carved from Workspace::pf (device pointers).
struct PrefillPtrs {
  int* hdr;          // [0] blocks, [1] shared-expert blocks
  PBlk* blk;         // block table
  uint16_t* xc;      // packed activations, core-matrix order, K permuted
  float* sx;         // per block: [H/64 groups][np] sums of x over each group
  uint16_t* hc_hi;   // packed SwiGLU outputs, bf16 high part
  uint16_t* hc_lo;   // bf16 low part (h - hi)
  float* sh;         // per block: [F/64 groups][np] sums of h over each group
  float* y_pair;     // [T*k][H] routed expert outputs, grouped pair order
  float* y_sh;       // [T][H] shared expert outputs
  int* inv;          // [T*k] grouped pair position of (token, rank)
};

struct LayerArgs {
  int H, E, k, F, Fs, T;
  const uint8_t* records;  // E records at `stride` (or the residency slot pool)
  const uint8_t* shared;   // shared record or null
  const uint8_t* rcodes;   // router codes [E][H]
  const uint32_t* rsb;     // router sb words [E][H/64]
  const float* beta;       // [E] or null
  const uint16_t* cbs;     // 3-bit residual-VQ experts: codebooks [3 kinds][3 stages][256][8]
                           // bf16 (kinds gate, up, down); null for 4-bit affine experts
  const int32_t* slot_of;  // [E] expert -> slot (residency) or null for identity
  const int32_t* slot_tag; // [n_slots] expert id held by each slot, or null
  int n_slots;             // slots of the pool when slot_of is set
  const uint16_t* x;       // [T][H] bf16
  uint16_t* out_bf16;      // [T][H]
  float* out_f32;          // [T][H] or null
  int32_t* ids;            // [T][k]
  float* weights;          // [T][k]
  int32_t* ids_host;       // [T][k] copies of ids and weights in mapped page-locked host
  float* weights_host;     // memory (the router writes both), or null
  Workspace ws;
  RecordOffsets off_r, off_s;  // layouts for F and Fs
  // per-launch geometry (plan_decode / plan_prefill)
  int gu_nrl;                  // gate|up row-lanes; an item holds 2*gu_nrl gate + up rows
  int gu_stage, gu_nst;        // gate|up stage bytes and stage count
  int gu_rows;                 // single-token gate|up: rows per thread per item (4 or 8)
  int gu_part;                 // single-token gate|up items: 0 all, 1 shared expert only,
                               // 2 routed experts only
  int dn_rt, dn_tiles;         // down row tile and number of tiles (H / dn_rt)
  int dn_stage, dn_nst;        // down stage bytes and stage count
  int f1_rt, f1_stage, f1_nst; // fused single-token kernel: down rows per item, stage bytes
                               // and count (f1_nst == 0: not planned)
  PrefillPtrs pf;              // prefill chunk scratch (tensor-core path)
  int xq_nconv;                // router CTAs after the logits CTAs that write ws.xq (0: none)
  int x_pdl;                   // x is written by the kernel launched just before the single-
                               // token router (the host entry's staging kernel): the router is
                               // its programmatic dependent and waits for it before reading x
  int prof_on;                 // record prof[] events between kernels, no PDL
  void* prof[4];               // cudaEvent_t: before router / gate|up / down, after down
};

}  // namespace moe
