/*
 * oracle.c -- plain, slow, single-threaded fp64 statement of the MoE FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path links,
 * loads or calls this file.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark may use it.  It shares no code, header,
 * table or helper with the CUDA library: it re-derives the record layout
 * and every formula on its own from the pages it cites.
 *
 * What it computes, per token x (bf16, widened exactly to double):
 *
 *   1. dequantisation of "MLX affine" weights, 4-bit (experts) or 8-bit
 *      (router), group 64 along the input dimension:
 *          w[r][j] = s[r][j/64] * q[r][j] + b[r][j/64]
 *      -- TurboFieldfare page, section "Belleği azaltan çalışma yapısı"
 *         (affine 4-bit group 64, 8-bit router, 4-bit shared and routed
 *         experts).  Reading: "affine" is scale*code + bias (MLX), not
 *         scale*(code - zero).
 *   2. router logits l_e = sum_j W_r[e][j] x_j + beta_e
 *      -- same page, section "Token üretim süreci" (the router runs on the
 *         GPU from resident weights).  beta is an optional per-expert logit
 *         offset (0 when absent) used only to shape synthetic workloads.
 *   3. top-k: order experts by (l descending, id ascending) and keep the
 *      first k -- same section (the router's best 8 ids per layer).
 *   4. weights p_i = exp(l_i - l_max) / sum_{j in top-k} exp(l_j - l_max),
 *      i.e. a softmax over all experts renormalised over the top-k (which is
 *      the same number as a softmax over the top-k logits alone).
 *   5. expert FFN: g = W_g x, u = W_u x, h = silu(g) * u, y = W_d h with
 *      silu(z) = z / (1 + exp(-z)).  gate, up and down live contiguously in
 *      one record -- WASTE page ("Kimi K3'ü 29 GB RAM'de ..."), section
 *      "Disk streaming mimarisi" (gate, up, down adjacent, one read).
 *   6. combine: out = y_shared + sum_i p_i * y_{e_i}; the shared branch has
 *      weight 1 -- TurboFieldfare page, section "Token üretim süreci"
 *      (shared output and routed output are combined).
 *
 * Record format (this library's own choice; the pages fix only that gate,
 * up and down are adjacent and records are 4 KiB aligned):
 *   [gate codes F x H/2][up codes F x H/2][down codes H x F/2]
 *   [gate sb F x H/64][up sb F x H/64][down sb H x F/64]
 *   codes: row-major [out][in], element j of a row in byte j/2, low nibble
 *          when j is even;
 *   sb:    one little-endian 32-bit word per (row, group): bits 0..15 the
 *          bf16 scale, bits 16..31 the bf16 bias;
 *   stride: total size rounded up to 4096 bytes.
 * Router: codes u8 [E][H] row-major, sb words [E][H/64] as above.
 *
 * Second expert format, 3-bit residual VQ -- WASTE page, section
 * "Quantization ve doğruluk": each run of 8 weights along a row is the sum
 * of one codeword from each of 3 stages, every stage a codebook of 256
 * eight-value codewords, so 3 code bytes per 8 weights (3.00 bits/weight):
 *     w[r][8b + i] = C1[q1(r,b)][i] + C2[q2(r,b)][i] + C3[q3(r,b)][i]
 * Readings where the page is silent: the codebooks are per layer and matrix
 * kind (gate, up, down), kept with the router rather than in the records
 * (the page's codebooks sit outside the checksummed expert records);
 * codewords are bf16; there is no scale or bias.  Record: [gate codes
 * F x 3H/8][up codes F x 3H/8][down codes H x 3F/8], row-major, a row's
 * blocks in order and each block's three stage bytes in stage order; stride
 * rounded up to 4096.  Codebooks: bf16 [kind][stage][256][8].
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORC_GROUP 64

/* ---- bf16 ---------------------------------------------------------------- */

/* A bf16 value is the top half of an IEEE binary32; widening is exact. */
double orc_bf16_to_double(uint16_t h)
{
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ---- record layout ------------------------------------------------------- */

typedef struct {
    uint64_t gate_codes, up_codes, down_codes; /* byte offsets */
    uint64_t gate_sb, up_sb, down_sb;          /* byte offsets */
    uint64_t bytes;                            /* unpadded size */
    uint64_t stride;                           /* bytes rounded up to 4096 */
} orc_layout;

void orc_record_layout(int H, int F, orc_layout *L)
{
    uint64_t h = (uint64_t)H, f = (uint64_t)F;
    uint64_t mat_codes = f * h / 2;           /* gate or up, also down */
    uint64_t mat_sb = f * (h / ORC_GROUP) * 4; /* gate or up */
    uint64_t down_sb = h * (f / ORC_GROUP) * 4;
    L->gate_codes = 0;
    L->up_codes = mat_codes;
    L->down_codes = 2 * mat_codes;
    L->gate_sb = 3 * mat_codes;
    L->up_sb = L->gate_sb + mat_sb;
    L->down_sb = L->up_sb + mat_sb;
    L->bytes = L->down_sb + down_sb;
    L->stride = (L->bytes + 4095u) / 4096u * 4096u;
}

/* ---- dequantisation ------------------------------------------------------ */

static uint32_t load_u32_le(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
           ((uint32_t)p[3] << 24);
}

/* Weight (r, j) of a 4-bit matrix with `cols` inputs: s*q + b (step 1). */
double orc_dequant4(const uint8_t *codes, const uint8_t *sb, int cols, int r, int j)
{
    size_t row_bytes = (size_t)cols / 2;
    uint8_t byte = codes[(size_t)r * row_bytes + (size_t)j / 2];
    int q = (j % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
    uint32_t w = load_u32_le(sb + ((size_t)r * (cols / ORC_GROUP) + j / ORC_GROUP) * 4);
    double s = orc_bf16_to_double((uint16_t)(w & 0xFFFFu));
    double b = orc_bf16_to_double((uint16_t)(w >> 16));
    return s * (double)q + b;
}

/* Weight (r, j) of the 8-bit router matrix: s*q + b (step 1). */
double orc_dequant8(const uint8_t *codes, const uint8_t *sb, int cols, int r, int j)
{
    int q = codes[(size_t)r * cols + j];
    uint32_t w = load_u32_le(sb + ((size_t)r * (cols / ORC_GROUP) + j / ORC_GROUP) * 4);
    double s = orc_bf16_to_double((uint16_t)(w & 0xFFFFu));
    double b = orc_bf16_to_double((uint16_t)(w >> 16));
    return s * (double)q + b;
}

/* y[r] = sum_j W[r][j] x[j] for a 4-bit matrix, one weight at a time. */
void orc_gemv4(const uint8_t *codes, const uint8_t *sb, int rows, int cols,
               const double *x, double *y)
{
    for (int r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int j = 0; j < cols; ++j)
            acc += orc_dequant4(codes, sb, cols, r, j) * x[j];
        y[r] = acc;
    }
}

/* ---- 3-bit residual VQ (second expert format) ----------------------------- */

void orc_rvq_layout(int H, int F, orc_layout *L)
{
    uint64_t mat = (uint64_t)F * (uint64_t)H / 8u * 3u; /* gate, up or down codes */
    L->gate_codes = 0;
    L->up_codes = mat;
    L->down_codes = 2 * mat;
    L->bytes = 3 * mat;
    L->gate_sb = L->up_sb = L->down_sb = L->bytes; /* no scale/bias words */
    L->stride = (L->bytes + 4095u) / 4096u * 4096u;
}

/* Weight (r, j) of an RVQ matrix with `cols` inputs; cb is one kind's
 * codebooks [3][256][8]. */
double orc_dequant_rvq(const uint8_t *codes, const uint16_t *cb, int cols, int r, int j)
{
    const uint8_t *blk = codes + (size_t)r * ((size_t)cols / 8 * 3) + (size_t)(j / 8) * 3;
    double w = 0.0;
    for (int s = 0; s < 3; ++s)
        w += orc_bf16_to_double(cb[((size_t)s * 256 + blk[s]) * 8 + (size_t)(j % 8)]);
    return w;
}

void orc_gemv_rvq(const uint8_t *codes, const uint16_t *cb, int rows, int cols,
                  const double *x, double *y)
{
    for (int r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int j = 0; j < cols; ++j)
            acc += orc_dequant_rvq(codes, cb, cols, r, j) * x[j];
        y[r] = acc;
    }
}

/* ---- router, top-k, weights (steps 2-4) ---------------------------------- */

void orc_router_logits(const uint8_t *codes, const uint8_t *sb, const float *beta,
                       int E, int H, const double *x, double *logits)
{
    for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int j = 0; j < H; ++j)
            acc += orc_dequant8(codes, sb, H, e, j) * x[j];
        logits[e] = acc + (beta ? (double)beta[e] : 0.0);
    }
}

/* Top-k by (logit descending, id ascending); ids in that order.  `taken` is
 * caller scratch of E bytes. */
void orc_topk(const double *logits, int E, int k, int32_t *ids, double *p,
              unsigned char *taken)
{
    memset(taken, 0, (size_t)E);
    for (int i = 0; i < k; ++i) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            if (best < 0 || logits[e] > logits[best])
                best = e; /* strict '>' keeps the lower id on ties */
        }
        taken[best] = 1;
        ids[i] = best;
    }
    double lmax = logits[ids[0]];
    double z = 0.0;
    for (int i = 0; i < k; ++i)
        z += exp(logits[ids[i]] - lmax);
    for (int i = 0; i < k; ++i)
        p[i] = exp(logits[ids[i]] - lmax) / z;
}

/* ---- expert FFN (step 5) ------------------------------------------------- */

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* y[H] = W_d (silu(W_g x) * (W_u x)) for one record with ffn width F.
 * scratch must hold 3*F doubles. */
void orc_expert(const uint8_t *rec, int H, int F, const double *x, double *y,
                double *scratch)
{
    orc_layout L;
    orc_record_layout(H, F, &L);
    double *g = scratch, *u = scratch + F, *h = scratch + 2 * F;
    orc_gemv4(rec + L.gate_codes, rec + L.gate_sb, F, H, x, g);
    orc_gemv4(rec + L.up_codes, rec + L.up_sb, F, H, x, u);
    for (int j = 0; j < F; ++j)
        h[j] = orc_silu(g[j]) * u[j];
    orc_gemv4(rec + L.down_codes, rec + L.down_sb, H, F, h, y);
}

/* The same expert in the RVQ format; cbs = the layer's codebooks
 * [gate, up, down][3][256][8]. */
void orc_expert_rvq(const uint8_t *rec, const uint16_t *cbs, int H, int F, const double *x,
                    double *y, double *scratch)
{
    orc_layout L;
    orc_rvq_layout(H, F, &L);
    const size_t kind = 3 * 256 * 8;
    double *g = scratch, *u = scratch + F, *h = scratch + 2 * F;
    orc_gemv_rvq(rec + L.gate_codes, cbs, F, H, x, g);
    orc_gemv_rvq(rec + L.up_codes, cbs + kind, F, H, x, u);
    for (int j = 0; j < F; ++j)
        h[j] = orc_silu(g[j]) * u[j];
    orc_gemv_rvq(rec + L.down_codes, cbs + 2 * kind, H, F, h, y);
}

/* ---- whole layer for one token (steps 1-6) ------------------------------- */

typedef struct {
    int H, E, k, F, Fs;             /* Fs == 0: no shared expert */
    const uint8_t *const *records;  /* E pointers; unselected may be NULL */
    const uint8_t *shared_record;   /* NULL when Fs == 0 */
    const uint8_t *router_codes;    /* [E][H] */
    const uint8_t *router_sb;       /* [E][H/64] words */
    const float *beta;              /* [E] or NULL */
    const uint16_t *codebooks;      /* RVQ experts: [3][3][256][8] bf16; NULL: 4-bit affine */
} orc_layer;

static void layer_expert(const orc_layer *Ly, const uint8_t *rec, int F, const double *x,
                         double *y, double *scratch)
{
    if (Ly->codebooks)
        orc_expert_rvq(rec, Ly->codebooks, Ly->H, F, x, y, scratch);
    else
        orc_expert(rec, Ly->H, F, x, y, scratch);
}

/* Route one token: logits (E doubles), ids (k), p (k).  taken: E bytes. */
void orc_route(const orc_layer *Ly, const uint16_t *x_bf16, double *xd,
               double *logits, int32_t *ids, double *p, unsigned char *taken)
{
    for (int j = 0; j < Ly->H; ++j)
        xd[j] = orc_bf16_to_double(x_bf16[j]);
    orc_router_logits(Ly->router_codes, Ly->router_sb, Ly->beta, Ly->E, Ly->H, xd,
                      logits);
    orc_topk(logits, Ly->E, Ly->k, ids, p, taken);
}

/* Full layer for one token.  Returns 0, or -1 when a selected expert's
 * record pointer is NULL.  work must hold H + E + H + 3*max(F,Fs) doubles,
 * taken E bytes. */
int orc_moe_token(const orc_layer *Ly, const uint16_t *x_bf16, double *out,
                  int32_t *ids, double *p, double *work, unsigned char *taken)
{
    int H = Ly->H;
    double *xd = work, *logits = work + H, *y = logits + Ly->E, *scr = y + H;
    orc_route(Ly, x_bf16, xd, logits, ids, p, taken);
    for (int r = 0; r < H; ++r)
        out[r] = 0.0;
    if (Ly->Fs > 0) {
        layer_expert(Ly, Ly->shared_record, Ly->Fs, xd, y, scr);
        for (int r = 0; r < H; ++r)
            out[r] = y[r];
    }
    for (int i = 0; i < Ly->k; ++i) {
        const uint8_t *rec = Ly->records[ids[i]];
        if (!rec)
            return -1;
        layer_expert(Ly, rec, Ly->F, xd, y, scr);
        for (int r = 0; r < H; ++r)
            out[r] += p[i] * y[r];
    }
    return 0;
}

/* ---- dense masked evaluation (for the brute-force pin) ------------------- */

/* Evaluates EVERY expert densely and combines with a mask built from the
 * top-k set: out = y_shared + sum_e [e in topk] * p_e * y_e.  Same maths as
 * orc_moe_token but a different order of work; used by the tests only to
 * pin the sparse path.  records must all be non-NULL. */
int orc_moe_token_dense(const orc_layer *Ly, const uint16_t *x_bf16, double *out,
                        double *work, unsigned char *taken, int32_t *ids, double *p)
{
    int H = Ly->H, E = Ly->E;
    double *xd = work, *logits = work + H, *y = logits + E, *scr = y + H;
    orc_route(Ly, x_bf16, xd, logits, ids, p, taken);
    for (int r = 0; r < H; ++r)
        out[r] = 0.0;
    for (int e = 0; e < E; ++e) {
        double pe = 0.0;
        for (int i = 0; i < Ly->k; ++i)
            if (ids[i] == e)
                pe = p[i];
        if (!Ly->records[e])
            return -1;
        layer_expert(Ly, Ly->records[e], Ly->F, xd, y, scr);
        for (int r = 0; r < H; ++r)
            out[r] += pe * y[r];
    }
    if (Ly->Fs > 0) {
        layer_expert(Ly, Ly->shared_record, Ly->Fs, xd, y, scr);
        for (int r = 0; r < H; ++r)
            out[r] += y[r];
    }
    return 0;
}

/* ---- LFU residency policy (host bookkeeping, replayed from an id stream) --
 * TurboFieldfare page, section "Token üretim süreci": the chosen ids are
 * checked against a bounded per-layer LFU cache and misses are filled.
 * Readings where the page says only "LFU": use counts are per expert per
 * layer and cumulative over the run (kept for evicted experts too); the
 * victim is the resident, unpinned expert with the lowest count, ties to the
 * least recently used, then to the lower id; every expert the current step
 * needs is pinned; a miss costs one full record copy.
 *
 * State arrays (caller-owned, zeroed before the first step):
 *   slot_expert[n_slots] (-1 = empty), count[E], last_use[E]
 * For one step with ids[k] (distinct), writes hit[k] (1/0) and slot[k] and
 * returns the number of misses.  step is the 1-based step number.  */
int orc_lfu_step(int n_slots, int E, int *slot_expert, int64_t *count,
                 int64_t *last_use, const int32_t *ids, int k, int64_t step,
                 int *hit, int *slot)
{
    int misses = 0;
    for (int i = 0; i < k; ++i) {
        count[ids[i]] += 1;
        last_use[ids[i]] = step;
    }
    for (int i = 0; i < k; ++i) {
        int found = -1;
        for (int s = 0; s < n_slots; ++s)
            if (slot_expert[s] == ids[i])
                found = s;
        hit[i] = found >= 0;
        slot[i] = found;
    }
    for (int i = 0; i < k; ++i) {
        if (hit[i])
            continue;
        ++misses;
        int victim = -1;
        for (int s = 0; s < n_slots && victim < 0; ++s)
            if (slot_expert[s] < 0)
                victim = s; /* lowest empty slot first */
        if (victim < 0) {
            for (int s = 0; s < n_slots; ++s) {
                int e = slot_expert[s];
                int pinned = 0;
                for (int t = 0; t < k; ++t)
                    if (ids[t] == e)
                        pinned = 1;
                if (pinned)
                    continue;
                if (victim < 0) {
                    victim = s;
                    continue;
                }
                int v = slot_expert[victim];
                if (count[e] < count[v] ||
                    (count[e] == count[v] &&
                     (last_use[e] < last_use[v] ||
                      (last_use[e] == last_use[v] && e < v))))
                    victim = s;
            }
        }
        if (victim < 0)
            return -1; /* more distinct ids than slots */
        slot_expert[victim] = ids[i];
        slot[i] = victim;
    }
    return misses;
}

/* ---- Router lookahead into the LFU cache ---------------------------------
 * WASTE page, section "Önceden okuma ve router tahmini": before a layer's own
 * hidden state exists, that layer's router is run on the hidden state one
 * residual earlier, and the first few experts of the predicted ranking are
 * read into the cache; the layer's own router still chooses the experts, so
 * the output does not change, only which reads are demand misses.
 * Readings where the page is silent:
 *   * the predictions of a batch are visited rank-major (every token's first
 *     choice, then every token's second, ...), repeats skipped;
 *   * every visited expert, resident or not, is pinned before any slot is
 *     chosen, and stays pinned until the layer's next demand step, so one
 *     prediction never evicts another;
 *   * a non-resident prediction takes the lowest empty slot, else evicts the
 *     unpinned resident with the lowest (use count, last use, id), as a
 *     demand miss does; when every slot is pinned it is dropped;
 *   * use counts and last-use steps are not touched: only demand steps use
 *     an expert.
 * pred[n] are the predicted ids already in visiting order (repeats allowed).
 * pinned[E] and fresh[E] are 0/1 arrays owned by the caller: pinned marks
 * the lookahead pins (the caller clears them at the next demand step), fresh
 * marks records this lookahead copied that no demand step has used yet.
 * Writes slot[n] (the slot the prediction occupies, -1 if dropped) and
 * *evictions; returns the number of records copied. */
int orc_lfu_lookahead(int n_slots, int E, int *slot_expert, const int64_t *count,
                      const int64_t *last_use, uint8_t *pinned, uint8_t *fresh,
                      const int32_t *pred, int n, int *slot, int *evictions)
{
    int copies = 0;
    *evictions = 0;
    for (int i = 0; i < n; ++i)
        pinned[pred[i]] = 1;
    for (int i = 0; i < n; ++i) {
        int e = pred[i], where = -1;
        for (int s = 0; s < n_slots; ++s)
            if (slot_expert[s] == e)
                where = s;
        if (where >= 0) {
            slot[i] = where;
            continue;
        }
        int victim = -1;
        for (int s = 0; s < n_slots && victim < 0; ++s)
            if (slot_expert[s] < 0)
                victim = s;
        if (victim < 0) {
            for (int s = 0; s < n_slots; ++s) {
                int r = slot_expert[s];
                if (pinned[r])
                    continue;
                if (victim < 0) {
                    victim = s;
                    continue;
                }
                int v = slot_expert[victim];
                if (count[r] < count[v] ||
                    (count[r] == count[v] &&
                     (last_use[r] < last_use[v] ||
                      (last_use[r] == last_use[v] && r < v))))
                    victim = s;
            }
            if (victim >= 0) {
                fresh[slot_expert[victim]] = 0;
                ++*evictions;
            }
        }
        slot[i] = victim;
        if (victim < 0)
            continue; /* every slot pinned: dropped */
        slot_expert[victim] = e;
        fresh[e] = 1;
        ++copies;
    }
    return copies;
}
