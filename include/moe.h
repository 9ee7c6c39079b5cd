/*
 * moe.h -- C ABI of a GB300 (sm_103a) Mixture-of-Experts FFN layer.
 *
 * The layer, per token x (bf16, H values):
 *   1. router: logits l_e = sum_j W_r[e][j] x_j + beta_e over E experts, W_r
 *      8-bit affine with one bf16 (scale, bias) per 64 inputs;
 *   2. top-k by (logit descending, expert id ascending), weights
 *      p_i = softmax over all experts renormalised over the k chosen ones;
 *   3. for every chosen expert and the always-resident shared expert:
 *      h = silu(W_g x) * (W_u x), y = W_d h, with W_g, W_u, W_d 4-bit affine,
 *      group 64 along the input dimension;
 *   4. out = y_shared + sum_i p_i y_{e_i}.
 * Sources: TurboFieldfare page ("Gemma 4 26B'yi 2GB RAM ile çalıştıran açık
 * kaynak motor"), sections "Belleği azaltan çalışma yapısı" (MLX affine
 * 4-bit group 64 experts, 8-bit router) and "Token üretim süreci" (router on
 * the GPU, top-8 ids against a bounded LFU cache, shared expert computed
 * while misses are read, shared and routed outputs combined, prompt prefill
 * in chunks of at most 128 tokens so one fetched expert serves several
 * rows); WASTE page ("Kimi K3'ü 29 GB RAM'de ..."), section "Disk streaming
 * mimarisi" (gate, up and down adjacent in one 4 KiB-aligned expert record).
 *
 * Conventions for every call:
 *   - Return 0 (MOE_OK) or a negative MOE_ERR_* code; moe_last_error()
 *     gives a thread-local message for the last failing call.
 *   - "device" pointers are CUDA global-memory addresses on the current
 *     device; "host" pointers are CPU addresses (pinned for best copy speed).
 *   - The caller owns every device and host buffer: weights, activations,
 *     outputs, workspace and slot pools.  A moe_layer handle stores pointers
 *     and shapes only; moe_close frees host bookkeeping only.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *     Device work is asynchronous on it; argument errors are detected on the
 *     host before any launch.  Errors raised by device code (MOE_ERR_TIMEOUT,
 *     MOE_ERR_RESIDENCY) are latched in the workspace and returned by
 *     moe_check().
 *   - Device pointers must be 16-byte aligned (MOE_ERR_ALIGN otherwise);
 *     expert records additionally start on 256-byte boundaries.
 *   - Hidden-state magnitudes must stay below 2^40 (the GEMV kernels pre-
 *     scale activations by powers of two up to 2^85); NaN/Inf inputs are
 *     outside the contract.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    MOE_OK = 0,
    MOE_ERR_ARG = -1,         /* bad shape, size, null pointer, wrong handle */
    MOE_ERR_ALIGN = -2,       /* pointer not 16-byte (records: 256-byte) aligned */
    MOE_ERR_CUDA = -3,        /* a CUDA runtime call failed; see moe_last_error() */
    MOE_ERR_TIMEOUT = -4,     /* a bounded device-side wait expired */
    MOE_ERR_RESIDENCY = -5,   /* a slot's expert tag did not match the routed id */
    MOE_ERR_NOMEM = -6,       /* host bookkeeping allocation failed */
    MOE_ERR_UNSUPPORTED = -7  /* device is not sm_103 or lacks resources */
};

/* Shapes and quantisation of one layer.  Limits: hidden H in [64, 8192] and a
 * multiple of 64; n_experts E in [1, 1024]; top_k in [1, min(E, 32)]; ffn F
 * and shared_ffn Fs multiples of 64 in [64, 8192] (Fs = 0: no shared
 * expert); group must be 64; wbits 4 (affine experts, moe_record_layout) or
 * 3 (residual-VQ experts, moe_rvq_record_layout_of); rbits 8; max_tokens in
 * [1, 128] bounds B for decode and T for prefill chunks. */
typedef struct moe_layer_desc {
    int32_t hidden;
    int32_t n_experts;
    int32_t top_k;
    int32_t ffn;
    int32_t shared_ffn;
    int32_t group;
    int32_t wbits;
    int32_t rbits;
    int32_t max_tokens;
} moe_layer_desc;

/* Byte offsets of the regions of one expert record with FFN width F:
 *   [gate codes F x H/2][up codes F x H/2][down codes H x F/2]
 *   [gate sb F x H/64][up sb F x H/64][down sb H x F/64]
 * Codes are row-major [out][in], element j of a row in byte j/2, low nibble
 * for even j.  One little-endian 32-bit "sb" word per (row, group of 64
 * inputs): bits 0..15 the bf16 scale s, bits 16..31 the bf16 bias b, so
 * w = s*q + b.  `stride` is `bytes` rounded up to 4096. */
typedef struct moe_record_layout {
    uint64_t gate_codes, up_codes, down_codes;
    uint64_t gate_sb, up_sb, down_sb;
    uint64_t bytes;
    uint64_t stride;
} moe_record_layout;

/* Device weights of one layer (all caller-owned, read-only to the library).
 *   expert_records: E records back to back at stride moe_expert_bytes(ffn);
 *                   may be NULL for a layer used only through the residency
 *                   API, whose slot pool then holds the records.
 *   shared_record:  one record with FFN width shared_ffn (NULL iff Fs == 0).
 *   router_codes:   uint8 [E][H], one 8-bit code per weight.
 *   router_sb:      uint32 [E][H/64] sb words as in moe_record_layout.
 *   router_logit_bias: float [E] added to the logits, or NULL for none.
 *   expert_codebooks: wbits = 3 only (NULL otherwise): bf16 [3][3][256][8],
 *                   the layer's residual-VQ codebooks for gate, up and down,
 *                   3 stages each, 256 codewords of 8 values (16-byte
 *                   aligned).  WASTE page, section "Quantization ve
 *                   doğruluk": each run of 8 weights along a row is the sum
 *                   of one codeword per stage, named by 3 code bytes. */
typedef struct moe_layer_weights {
    const void *expert_records;
    const void *shared_record;
    const uint8_t *router_codes;
    const uint32_t *router_sb;
    const float *router_logit_bias;
    const uint16_t *expert_codebooks;
} moe_layer_weights;

typedef struct moe_layer moe_layer;

/* Record layout for hidden H and FFN width F (see moe_record_layout).
 * Returns MOE_ERR_ARG for shapes outside the limits above. */
int moe_record_layout_of(int32_t hidden, int32_t ffn, moe_record_layout *out);

/* Record layout of a residual-VQ expert (wbits = 3): code bytes only,
 *   [gate codes F x 3H/8][up codes F x 3H/8][down codes H x 3F/8]
 * row-major; a row holds its blocks of 8 inputs in order, each block 3 bytes
 * (the codeword index of stage 1, 2, 3).  The sb offsets equal `bytes` (no
 * scale/bias words); `stride` is `bytes` rounded up to 4096.  Decode and the
 * expert cache (which copies these records); moe_prefill_chunk needs
 * wbits = 4. */
int moe_rvq_record_layout_of(int32_t hidden, int32_t ffn, moe_record_layout *out);

/* Stride in bytes of one expert record of width `ffn` in desc's format
 * (0 on bad shapes). */
size_t moe_expert_bytes(const moe_layer_desc *desc, int32_t ffn);

/* Validates shapes and pointers, queries the device (must be sm_103) and
 * returns a handle.  No device allocation, no device work. */
int moe_open(const moe_layer_desc *desc, const moe_layer_weights *weights, moe_layer **out);

/* Frees the handle (host memory only).  NULL is accepted. */
void moe_close(moe_layer *layer);

/* Bytes of device workspace that calls with up to `max_tokens` tokens need
 * (0 on a bad handle or size).  One workspace must not be used by two calls
 * that overlap on the GPU. */
size_t moe_workspace_bytes(const moe_layer *layer, int32_t max_tokens);

/* Zero-fills a workspace (cudaMemsetAsync on `stream`).  Required once
 * before the first call that uses it; the library keeps its counters at
 * zero between calls afterwards. */
int moe_workspace_init(const moe_layer *layer, void *workspace, size_t workspace_bytes,
                       void *stream);

/* Decode step for B tokens (1 <= B <= max_tokens), all experts resident.
 *   x:        device bf16 [B][H] hidden states.
 *   out_bf16: device bf16 [B][H], round-to-nearest-even of the fp32 result.
 *   out_f32:  device float [B][H] or NULL.
 *   ids:      device int32 [B][k] chosen experts, by (logit desc, id asc).
 *   weights:  device float [B][k] routing weights (sum to 1 per token).
 * B == 0 returns MOE_OK and does nothing.  Fully asynchronous: no host sync. */
int moe_decode(moe_layer *layer, const uint16_t *x, int32_t B, uint16_t *out_bf16,
               float *out_f32, int32_t *ids, float *weights, void *workspace,
               size_t workspace_bytes, void *stream);

/* Prefill chunk of T tokens (1 <= T <= min(128, max_tokens)); same buffers and
 * semantics as moe_decode.  Expert work runs as a grouped GEMM on the 5th-gen
 * tensor cores (tcgen05, accumulators in tensor memory).  MOE_ERR_ARG on a
 * wbits = 3 layer. */
int moe_prefill_chunk(moe_layer *layer, const uint16_t *x, int32_t T, uint16_t *out_bf16,
                      float *out_f32, int32_t *ids, float *weights, void *workspace,
                      size_t workspace_bytes, void *stream);

/* moe_decode with HOST buffers: copies x in, runs the step, hands every
 * output back (out_f32_host may be NULL) and synchronises `stream` before it
 * returns.  Device staging lives in the workspace.  The layer keeps page-
 * locked input and output buffers and a private stream (made by its first
 * moe_decode_host call, sized for max_tokens, freed by moe_close).  Both
 * buffers are mapped into the device's address space: x goes through the
 * input buffer, from which a small kernel copies it into the workspace (a
 * single-token router overlaps that copy as its programmatic dependent);
 * the kernels write the outputs into the output buffer directly (the router
 * writes ids and weights both to the workspace and there), from where they
 * go to the caller's buffers after the synchronisation.  The first call for
 * a given (workspace, B, out_f32_host set or not) runs plain launches and
 * then captures the step (copy kernel, layer kernels) into a CUDA graph;
 * later such calls replay it with one graph launch on `stream` (the layer
 * keeps the last 4).  The profiling hook always takes plain
 * launches.  Calls on one layer from several threads are serialised by a
 * lock. */
int moe_decode_host(moe_layer *layer, const uint16_t *x_host, int32_t B,
                    uint16_t *out_bf16_host, float *out_f32_host, int32_t *ids_host,
                    float *weights_host, void *workspace, size_t workspace_bytes,
                    void *stream);

/* Synchronises `stream`, then reads the error word that device code latches
 * in `workspace`: MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_RESIDENCY.  After an
 * error it zeroes the workspace's persistent control block (error word and
 * the claim and completion counters a step that gave up may leave mid-count),
 * so the workspace is ready for the next call. */
int moe_check(const moe_layer *layer, void *workspace, void *stream);

/* Number of kernels one moe_decode call with B tokens launches on this
 * layer, as its dispatch would choose them (with a workspace sized for B):
 * 2 for one token on the fused single-token kernel (router, fused gate|up +
 * down), 3 where the single-token kernels are not fused; 3 for 2..16 tokens
 * on the few-token fused kernel (router, fused kernel, combine); B times the
 * single-token count for larger batches run one token at a time, 5 for the
 * tensor-core chunk kernels and 3 for the grouped kernels; 4 on a wbits = 3
 * layer (the router, then gate|up, down and combine for every token at
 * once).  0 for B = 0; -1 on a bad handle or B outside [0, max_tokens].
 * Host-only: no device work. */
int32_t moe_decode_kernels(const moe_layer *layer, int32_t B);

/* Profiling hook.  With `events` pointing to four cudaEvent_t (passed as
 * void*), later moe_decode / moe_prefill_chunk calls on this layer record
 * events[0] before the router kernel, events[1] before the first expert
 * kernel (gate|up, the fused kernel or the grouped GEMM), events[2] before
 * the second (down, the few-token combine, or right after the single-token
 * fused kernel, which has none) and events[3] after the last, and launch
 * without programmatic dependent launch so the intervals are per kernel.
 * NULL switches the hook off.  The events stay caller-owned. */
int moe_set_profile_events(moe_layer *layer, void *const *events);

/* Thread-local description of the last error (never NULL). */
const char *moe_last_error(void);

/* ---- Expert residency: a bounded HBM cache of expert records ---------------
 * TurboFieldfare page, section "Token üretim süreci": the router's chosen ids
 * are checked against a per-layer LFU cache of bounded size; misses are
 * filled from the slower tier while the shared expert is computed; shared
 * and routed outputs are combined when the reads finish.  Here the slow tier
 * is page-locked host memory holding all E records of the layer (same
 * record format and stride as moe_record_layout_of), the cache is a pool of
 * n_slots record slots in HBM, and misses are copied with cudaMemcpyAsync on
 * a caller-given copy stream.
 *
 * Policy: one use count per expert, cumulative over the run (kept after
 * eviction); all experts of the step are counted and pinned first; a miss
 * takes the lowest empty slot, else evicts the unpinned resident with the
 * lowest count, ties to the least recently used, then the lower id; experts
 * are visited in the order they first appear in the step's ids (token-major,
 * rank order).  A miss copies one whole record. */
typedef struct moe_residency moe_residency;

typedef struct {
    uint64_t steps;      /* cache steps: one per moe_residency_decode call, one per wave */
    uint64_t hits;       /* distinct experts of a step already resident */
    uint64_t misses;     /* distinct experts copied in */
    uint64_t evictions;  /* copies (misses or lookahead) that replaced a resident expert */
    uint64_t bytes_h2d;  /* record bytes copied host -> device for misses */
    uint64_t lookaheads;        /* moe_residency_lookahead calls that reached the cache */
    uint64_t lookahead_copies;  /* records copied in by a lookahead */
    uint64_t lookahead_hits;    /* hits on a record a lookahead copied, before any step used it */
    uint64_t lookahead_bytes;   /* record bytes copied host -> device by lookaheads */
} moe_residency_stats_t;

/* Host-side fault injection for tests (no device fault is involved). */
#define MOE_RESIDENCY_FAULT_NONE 0
#define MOE_RESIDENCY_FAULT_TAG 1   /* next step uploads a wrong tag for one of its slots:
                                       the kernels latch MOE_ERR_RESIDENCY (moe_check) */
#define MOE_RESIDENCY_FAULT_COPY 2  /* the next record copy (of a step or a lookahead) fails
                                       as if the copy had: MOE_ERR_CUDA, the slot is left
                                       empty */

/* Bytes of the device slot pool for n_slots slots: the records at the layer's
 * record stride, then the slot tables.  0 for an invalid handle or n_slots
 * outside [1, n_experts]. */
size_t moe_residency_pool_bytes(const moe_layer *layer, int32_t n_slots);

/* Opens the cache.  host_records (host, page-locked, 16-byte aligned): the
 * layer's E expert records at the record stride, read by the copies;
 * device_pool (device, 256-byte aligned, >= moe_residency_pool_bytes): slot
 * storage, owned by the caller, written only by this cache.  n_slots in
 * [top_k, n_experts].  Allocates small pinned host buffers and a few
 * events, freed by moe_residency_close.  The layer may have been opened with
 * expert_records = NULL.  A wbits = 3 layer's records are its residual-VQ
 * records (moe_rvq_record_layout_of): a miss copies 3 bits per weight, and
 * the codebooks stay resident with the router. */
int moe_residency_open(moe_layer *layer, const void *host_records, int32_t n_slots,
                       void *device_pool, size_t device_pool_bytes, moe_residency **out);

/* One decode step through the cache: arguments and outputs as moe_decode,
 * plus the copy stream (cudaStream_t as void*; may equal main_stream, which
 * then forgoes the overlap).  Order of work: the router on main_stream; the
 * ids to the host; for B = 1 the shared expert's gate|up on main_stream; the
 * host waits for the ids (this call blocks until the router has finished),
 * updates the cache and issues one cudaMemcpyAsync per miss and one for the
 * slot tables on copy_stream; main_stream waits for them, then runs the
 * routed experts and the combine.  A call whose tokens need more distinct
 * experts than there are slots runs as waves: consecutive tokens, each wave
 * growing while its experts fit the slots, each a step of its own (its
 * router runs again).  MOE_ERR_RESIDENCY (returned) if the router's ids are
 * out of range; the cache state is then unchanged.  Device-side tag
 * mismatches are latched and reported by moe_check. */
int moe_residency_decode(moe_residency *res, const uint16_t *x, int32_t B, uint16_t *out_bf16,
                         float *out_f32, int32_t *ids, float *weights, void *workspace,
                         size_t workspace_bytes, void *main_stream, void *copy_stream);

/* Router lookahead (WASTE page, section "Önceden okuma ve router tahmini":
 * before a layer's own hidden state exists, its router is run on the hidden
 * state one residual earlier and the first few predicted experts are read
 * ahead; the layer's own router still chooses, so outputs do not change).
 *   x: device bf16 [B][hidden], the earlier hidden state (e.g. the previous
 *      layer's input); B in [0, max_tokens].
 *   n_ahead in [0, top_k]: experts taken from the head of each token's
 *      predicted ranking (0: no work).
 *   ids, weights: device [B][top_k], the predicted routing (written).
 *   workspace: a workspace of this layer (moe_workspace_init) that no kernel
 *      running at the same time uses; moe_check it for device errors.
 *   stream: where the router runs; the caller orders it after x is written.
 *      The call blocks until the predicted ids are on the host.
 *   copy_stream: where the records are copied.  The copies are ordered after
 *      the previous moe_residency_decode's kernels and the previous
 *      lookahead, whatever the streams; the next moe_residency_decode is
 *      ordered after them.
 * Policy: predictions are visited rank-major (every token's first, then
 * every token's second, ...), repeats skipped; all are pinned until the next
 * moe_residency_decode; a non-resident one takes a slot by the demand rule
 * (only lookahead pins count) and is dropped when every slot is pinned; use
 * counts and last-use steps are not changed.  Errors as for
 * moe_residency_decode (MOE_ERR_RESIDENCY for an out-of-range id or a record
 * failing its CRC-32 check, with the cache state unchanged; MOE_ERR_CUDA for a
 * failed copy, whose slot is left empty). */
int moe_residency_lookahead(moe_residency *res, const uint16_t *x, int32_t B, int32_t n_ahead,
                            int32_t *ids, float *weights, void *workspace, size_t workspace_bytes,
                            void *stream, void *copy_stream);

/* Counters since open. */
int moe_residency_stats(const moe_residency *res, moe_residency_stats_t *out);

/* The expert held by each slot (-1 = empty), host copy; n >= n_slots. */
int moe_residency_slots(const moe_residency *res, int32_t *slot_expert, int32_t n);

/* Arms one of the MOE_RESIDENCY_FAULT_* modes for the next step (one-shot). */
int moe_residency_set_fault(moe_residency *res, int32_t mode);

/* Optional payload check of the host records (WASTE page, section "Disk
 * streaming mimarisi": a crc32 of each record, off by default, worth running
 * once on records whose copy cannot be trusted).
 *   crc: host uint32 [n_experts], the expected moe_crc32 of each record's
 *        payload: its first `bytes` bytes (moe_record_layout_of(hidden, ffn);
 *        the padding up to the stride is not covered), copied; NULL switches
 *        the check off.
 * While on, a record is checked on the host before its first upload; a
 * mismatch makes moe_residency_decode return MOE_ERR_RESIDENCY with the
 * cache state unchanged (the message names the expert).  Records already
 * resident are checked by this call (MOE_ERR_RESIDENCY, check left off, on
 * a mismatch).  Each record is checked once per handle. */
int moe_residency_verify(moe_residency *res, const uint32_t *crc);

/* CRC-32 as in IEEE 802.3 and zlib (reflected polynomial 0xEDB88320,
 * all-ones preset, complemented result) of `bytes` host bytes at `data`.
 * moe_crc32("123456789", 9) == 0xCBF43926.  Host only; no device work. */
uint32_t moe_crc32(const void *data, size_t bytes);

/* Frees the host bookkeeping (pinned buffers, events); NULL is a no-op. */
void moe_residency_close(moe_residency *res);

/* ---- Decode without a caller-allocated workspace --------------------------
 * The pages describe no such call: it exists for callers that cannot
 * allocate device memory when they run a step -- a plain C host with no
 * device allocator of its own, or one that must not call cudaMalloc /
 * cudaFree while serving (both synchronise the whole device and stall every
 * other stream) or whose allocator has already handed all of HBM to its own
 * pool.
 *
 * moe_decode_noalloc computes exactly what moe_decode computes (same
 * kernels, same arguments minus the workspace), with the workspace taken
 * from a static device array of MOE_NOALLOC_SCRATCH_BYTES bytes inside this
 * library, one per device.  The call itself allocates nothing.
 *
 * Limit: moe_workspace_bytes(layer, B) must be <= MOE_NOALLOC_SCRATCH_BYTES
 * (16 MiB: for H=7168, E=512, top-16, F=Fs=2048 that is B <= 31); a larger B
 * is rejected with MOE_ERR_ARG before anything is launched, and
 * moe_last_error() says to use moe_decode with a caller-allocated
 * workspace.  The layer's device must be the current device (MOE_ERR_ARG
 * otherwise).
 *
 * First call per device: looks up the scratch's device address once (with
 * that device current) and zeroes the whole scratch on `stream`, ordered
 * before the step.  The scratch's control words (error word, the router's
 * completion counter, item claim counters, per-expert and per-row-tile
 * completion counters) must start at zero; every later step leaves them
 * ready for the next one.  Make this first call before any stream capture
 * begins.  The looked-up address is kept for the life of the process: do not
 * use this entry point on a device after cudaDeviceReset() of that device.
 *
 * All calls on one device share the one scratch: calls whose executions
 * overlap (different streams, different threads or different layers without
 * an ordering between them) race on it and give undefined results.  Issue
 * them on one stream, or order them with events.  Errors that device code
 * latches (a bounded wait that ran out) stay in the scratch until
 * moe_check_noalloc reads and clears them.
 *
 * Pointers, alignment, sizes and return codes otherwise as moe_decode. */
#define MOE_NOALLOC_SCRATCH_BYTES (16u << 20)
int moe_decode_noalloc(moe_layer *layer, const uint16_t *x, int32_t B, uint16_t *out_bf16,
                       float *out_f32, int32_t *ids, float *weights, void *stream);

/* moe_check for the static scratch of moe_decode_noalloc on the layer's
 * device (which must be current): synchronises `stream`, reads the error
 * word and returns MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_RESIDENCY or MOE_ERR_ARG
 * as moe_check does; after an error it zeroes the scratch's persistent
 * control block (error word, claim and completion counters that a step that
 * gave up may leave mid-count), so later no-alloc steps start clean.
 * MOE_OK when no no-alloc step has run on the device yet.  Allocates
 * nothing; it synchronises, so it must not be called during stream
 * capture.  The pages have no counterpart. */
int moe_check_noalloc(const moe_layer *layer, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
