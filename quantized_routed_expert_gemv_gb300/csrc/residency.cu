// residency.cu -- the HBM expert cache of include/moe.h (moe_residency_*).
//
// TurboFieldfare page, section "Token üretim süreci": each layer's chosen
// expert ids are checked against a bounded LFU cache, the misses are read
// from the slower tier while the GPU computes the resident shared-expert
// branch, and the shared and routed outputs are combined once the reads are
// done.  Here the slow tier is pinned host memory, the cache is a pool of
// record-sized slots in HBM, misses are copied with cudaMemcpyAsync on a side
// stream, and the shared expert's gate|up runs meanwhile.
//
// Policy (the pages say only "LFU"; these readings are pinned by a
// hand-worked trace in the tests):
//   * one use count per expert, cumulative over the run, kept after eviction;
//   * every expert the step needs is counted and pinned before lookup;
//   * a miss takes the lowest-numbered empty slot, else evicts the unpinned
//     resident with the lowest count, ties to the least recently used, then
//     to the lower expert id;
//   * experts are visited in the order they first appear in the step's ids
//     (token-major, each token's ids in rank order).
//
// Per step (one host thread, main stream M, copy stream C):
//   M: router -> ids copied to pinned host memory -> event
//   M: shared expert gate|up (single-token path)
//   host: waits for the ids event, updates the cache, and for each miss
//   C: cudaMemcpyAsync(slot, host record) ... then the slot tables; event
//   M: waits for C's event -> routed gate|up -> down + combine
// Every kernel that reads a routed record checks the slot's tag against the
// expert it wants and latches MOE_ERR_RESIDENCY on a mismatch (moe_check).
//
// Router lookahead (WASTE page, section "Önceden okuma ve router tahmini":
// before a layer's own hidden state exists, its router runs on the hidden
// state one residual earlier and the first few predicted experts are read
// ahead; the true router still picks the experts): moe_residency_lookahead
// runs this layer's router on the earlier hidden state, pins the first
// n_ahead predictions of each token (rank-major) until the next step and
// copies the missing ones into slots chosen by the miss rule above, with no
// use counted.  Ordering, whatever streams the caller gives:
//   lookahead copies  after  the previous step's routed kernels (ev_done)
//                            and the previous lookahead (ev_ahead);
//   a step's copies   after  the same two events.
// Slot-table images are pinned buffers used in turn; one is rewritten only
// after its previous upload has completed.
//
// Optional payload check (WASTE page, section "Disk streaming mimarisi": a
// crc32 of each record, off by default, worth running once on records of
// uncertain origin): with moe_residency_verify, a record's CRC-32 is
// computed on the host before its first upload and compared with the
// caller's value; a mismatch refuses the step, cache state unchanged.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "kernels.h"

namespace moe {
int report_error(int code, const char* msg);
int report_cuda(cudaError_t e, const char* what);
const moe_layer_desc* layer_desc(const moe_layer* L);
uint64_t layer_record_stride(const moe_layer* L);
uint64_t layer_record_bytes(const moe_layer* L);
int prepare_cached_decode(moe_layer* L, const uint16_t* x, int32_t B, uint16_t* ob, float* of,
                          int32_t* ids, float* wts, void* ws, size_t ws_bytes, const uint8_t* pool,
                          const int32_t* slot_of, const int32_t* slot_tag, int n_slots, LayerArgs* a,
                          bool* single, int* num_sms, const char* name);
int prepare_route(moe_layer* L, const uint16_t* x, int32_t B, int32_t* ids, float* wts, void* ws,
                  size_t ws_bytes, LayerArgs* a, bool* single, int* num_sms, const char* name);
cudaError_t launch_b1_router(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_b1_shared(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_b1_routed(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_decode_router(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_decode_experts(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_rvq_experts(const LayerArgs& a, int num_sms, cudaStream_t st);
}  // namespace moe

namespace {

constexpr uint32_t kResMagic = 0x52657331u;  // "Res1"
constexpr int kTabRing = 4;                  // pinned slot-table images used in turn

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

size_t tables_offset(uint64_t stride, int n_slots) { return round256(static_cast<size_t>(n_slots) * stride); }

size_t tables_bytes(int E, int n_slots) { return round256(static_cast<size_t>(E + n_slots) * 4); }

// CRC-32 as in IEEE 802.3 / zlib: reflected polynomial 0xEDB88320, register
// preset to all ones, result complemented.  Eight bytes per step with eight
// 256-entry tables: t[0] is the one-byte table, t[j][i] the remainder of byte
// i followed by j zero bytes.
uint32_t g_crc[8][256];
std::once_flag g_crc_once;

void crc_tables() {
  for (uint32_t i = 0; i < 256; ++i) {
    uint32_t c = i;
    for (int b = 0; b < 8; ++b) c = (c & 1u) ? (c >> 1) ^ 0xEDB88320u : c >> 1;
    g_crc[0][i] = c;
  }
  for (int j = 1; j < 8; ++j)
    for (uint32_t i = 0; i < 256; ++i) g_crc[j][i] = (g_crc[j - 1][i] >> 8) ^ g_crc[0][g_crc[j - 1][i] & 0xFFu];
}

uint32_t crc32_update(uint32_t crc, const uint8_t* p, size_t n) {
  std::call_once(g_crc_once, crc_tables);
  uint32_t c = ~crc;
  while (n >= 8) {
    // little-endian by construction: the bytes are combined explicitly
    const uint32_t lo = c ^ (static_cast<uint32_t>(p[0]) | static_cast<uint32_t>(p[1]) << 8 |
                             static_cast<uint32_t>(p[2]) << 16 | static_cast<uint32_t>(p[3]) << 24);
    const uint32_t hi = static_cast<uint32_t>(p[4]) | static_cast<uint32_t>(p[5]) << 8 |
                        static_cast<uint32_t>(p[6]) << 16 | static_cast<uint32_t>(p[7]) << 24;
    c = g_crc[7][lo & 0xFFu] ^ g_crc[6][(lo >> 8) & 0xFFu] ^ g_crc[5][(lo >> 16) & 0xFFu] ^ g_crc[4][lo >> 24] ^
        g_crc[3][hi & 0xFFu] ^ g_crc[2][(hi >> 8) & 0xFFu] ^ g_crc[1][(hi >> 16) & 0xFFu] ^ g_crc[0][hi >> 24];
    p += 8, n -= 8;
  }
  while (n--) c = (c >> 8) ^ g_crc[0][(c ^ *p++) & 0xFFu];
  return ~c;
}

}  // namespace

extern "C" uint32_t moe_crc32(const void* data, size_t bytes) {
  if (!data && bytes) return 0u;
  return crc32_update(0u, static_cast<const uint8_t*>(data), bytes);
}

struct moe_residency {
  uint32_t magic;
  moe_layer* layer;
  int E, k, n_slots, max_tokens;
  uint64_t stride, rec_bytes;
  const uint8_t* host;        // pinned: E records at `stride`
  uint8_t* pool;              // device: n_slots records, then the slot tables
  int32_t* d_tables;          // device: slot_of[E] | slot_tag[n_slots]
  int32_t* h_tab[kTabRing];   // pinned images of the slot tables, uploaded in turn
  cudaEvent_t ev_tab[kTabRing];
  bool tab_used[kTabRing];
  int tab_next;
  int32_t* h_ids;             // pinned: the step's ids [max_tokens][k]
  int32_t* h_pids;            // pinned: a lookahead's predicted ids [max_tokens][k]
  cudaEvent_t ev_ids, ev_copy, ev_pids;
  cudaEvent_t ev_done;        // main stream, after the last step's routed kernels
  cudaEvent_t ev_ahead;       // copy stream, after the last lookahead's copies
  // cache state (host)
  std::vector<int32_t> slot_expert;  // [n_slots] expert held, -1 = empty
  std::vector<int32_t> slot_of;      // [E] slot holding the expert, -1 = not resident
  std::vector<int64_t> count, last_use;
  std::vector<int64_t> pinned_at;    // [E] step that pinned the expert
  std::vector<int32_t> order;        // the step's distinct experts, first-appearance order
  std::vector<uint8_t> ahead;        // [E] pinned by a lookahead until the next step
  std::vector<int32_t> ahead_list;   // the experts with ahead[] set
  std::vector<uint8_t> fresh;        // [E] copied by a lookahead, not yet used by a step
  std::vector<int32_t> pred;         // a lookahead's predictions, visiting order
  int64_t step;
  moe_residency_stats_t stats;
  int fault;
  std::vector<uint32_t> crc_expect;  // [E] caller's CRC-32 per record; empty: no check
  std::vector<uint8_t> crc_checked;  // [E] the record passed its check
};

static bool res_valid(const moe_residency* R) { return R && R->magic == kResMagic; }

static void destroy(moe_residency* R);

extern "C" size_t moe_residency_pool_bytes(const moe_layer* layer, int32_t n_slots) {
  const moe_layer_desc* d = moe::layer_desc(layer);
  if (!d || n_slots < 1 || n_slots > d->n_experts) return 0;
  return tables_offset(moe::layer_record_stride(layer), n_slots) + tables_bytes(d->n_experts, n_slots);
}

extern "C" int moe_residency_open(moe_layer* layer, const void* host_records, int32_t n_slots,
                                  void* device_pool, size_t pool_bytes, moe_residency** out) {
  if (!out) return moe::report_error(MOE_ERR_ARG, "moe_residency_open: out is NULL");
  *out = nullptr;
  const moe_layer_desc* d = moe::layer_desc(layer);
  if (!d) return moe::report_error(MOE_ERR_ARG, "moe_residency_open: invalid layer handle");
  if (n_slots < 1 || n_slots > d->n_experts)
    return moe::report_error(MOE_ERR_ARG, "moe_residency_open: n_slots must be in [1, n_experts]");

  if (n_slots < d->top_k)
    return moe::report_error(MOE_ERR_ARG, "moe_residency_open: fewer slots than top_k: a step could never fit");
  if (!host_records || !device_pool)
    return moe::report_error(MOE_ERR_ARG, "moe_residency_open: host_records and device_pool are required");
  if (reinterpret_cast<uintptr_t>(device_pool) % 256 || reinterpret_cast<uintptr_t>(host_records) % 16)
    return moe::report_error(MOE_ERR_ALIGN,
                             "moe_residency_open: device_pool must be 256-byte and host_records 16-byte aligned");
  const size_t need = moe_residency_pool_bytes(layer, n_slots);
  if (pool_bytes < need) return moe::report_error(MOE_ERR_ARG, "moe_residency_open: device_pool is smaller than moe_residency_pool_bytes()");
  cudaPointerAttributes pa;
  cudaError_t e = cudaPointerGetAttributes(&pa, host_records);
  if (e != cudaSuccess || pa.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    return moe::report_error(MOE_ERR_ARG, "moe_residency_open: host_records must be page-locked host memory");
  }
  moe_residency* R = new (std::nothrow) moe_residency();
  if (!R) return moe::report_error(MOE_ERR_NOMEM, "moe_residency_open: out of host memory");
  R->layer = layer;
  R->E = d->n_experts, R->k = d->top_k, R->n_slots = n_slots, R->max_tokens = d->max_tokens;
  R->stride = moe::layer_record_stride(layer), R->rec_bytes = moe::layer_record_bytes(layer);
  R->host = static_cast<const uint8_t*>(host_records);
  R->pool = static_cast<uint8_t*>(device_pool);
  R->d_tables = reinterpret_cast<int32_t*>(R->pool + tables_offset(R->stride, n_slots));
  R->slot_expert.assign(n_slots, -1);
  R->slot_of.assign(R->E, -1);
  R->count.assign(R->E, 0);
  R->last_use.assign(R->E, 0);
  R->pinned_at.assign(R->E, 0);
  R->ahead.assign(R->E, 0);
  R->fresh.assign(R->E, 0);
  const size_t nid = static_cast<size_t>(R->max_tokens) * R->k;
  R->order.reserve(nid);
  R->ahead_list.reserve(nid);
  R->pred.reserve(nid);
  const size_t tb = static_cast<size_t>(R->E + n_slots) * 4;
  e = cudaSuccess;
  for (int i = 0; i < kTabRing && !e; ++i)
    if (!(e = cudaHostAlloc(&R->h_tab[i], tb, cudaHostAllocDefault)))
      e = cudaEventCreateWithFlags(&R->ev_tab[i], cudaEventDisableTiming);
  if (e || (e = cudaHostAlloc(&R->h_ids, nid * 4, cudaHostAllocDefault)) ||
      (e = cudaHostAlloc(&R->h_pids, nid * 4, cudaHostAllocDefault)) ||
      (e = cudaEventCreateWithFlags(&R->ev_ids, cudaEventDisableTiming)) ||
      (e = cudaEventCreateWithFlags(&R->ev_copy, cudaEventDisableTiming)) ||
      (e = cudaEventCreateWithFlags(&R->ev_pids, cudaEventDisableTiming)) ||
      (e = cudaEventCreateWithFlags(&R->ev_done, cudaEventDisableTiming)) ||
      (e = cudaEventCreateWithFlags(&R->ev_ahead, cudaEventDisableTiming))) {
    destroy(R);
    return moe::report_cuda(e, "moe_residency_open: pinned buffers / events");
  }
  for (int i = 0; i < R->E + n_slots; ++i) R->h_tab[0][i] = -1;
  if ((e = cudaMemcpy(R->d_tables, R->h_tab[0], tb, cudaMemcpyHostToDevice))) {
    destroy(R);
    return moe::report_cuda(e, "moe_residency_open: slot tables");
  }
  R->magic = kResMagic;
  *out = R;
  return MOE_OK;
}

// Victim slot for a copy: the lowest empty slot, else the unpinned resident
// with the lowest (count, last use, id); -1 if every slot is pinned.  A
// step's experts are pinned during the step; a lookahead's predictions until
// the next step (a lookahead sees only those pins).
static int choose_slot(const moe_residency* R, bool lookahead) {
  int best = -1;
  for (int s = 0; s < R->n_slots; ++s) {
    const int e = R->slot_expert[s];
    if (e < 0) return s;
    if (R->ahead[e] || (!lookahead && R->pinned_at[e] == R->step)) continue;
    if (best < 0) {
      best = s;
      continue;
    }
    const int b = R->slot_expert[best];
    const bool better = R->count[e] != R->count[b] ? R->count[e] < R->count[b]
                        : R->last_use[e] != R->last_use[b] ? R->last_use[e] < R->last_use[b]
                                                           : e < b;
    if (better) best = s;
  }
  return best;
}

// Where a step needs more distinct experts than there are slots, its tokens
// run in waves: a wave grows token by token while the union of its tokens'
// experts fits the slots.  Writes each wave's first token to starts.
static void plan_waves(const moe_residency* R, int B, std::vector<int>* starts) {
  std::vector<uint8_t> in(R->E, 0);
  std::vector<int32_t> members;
  starts->assign(1, 0);
  for (int t = 0; t < B; ++t) {
    const int32_t* row = R->h_ids + static_cast<size_t>(t) * R->k;
    int add = 0;
    for (int i = 0; i < R->k; ++i) add += in[row[i]] ? 0 : 1;
    if (static_cast<int>(members.size()) + add > R->n_slots) {
      for (int32_t e : members) in[e] = 0;
      members.clear();
      starts->push_back(t);
    }
    for (int i = 0; i < R->k; ++i)
      if (!in[row[i]]) in[row[i]] = 1, members.push_back(row[i]);
  }
}

// Uploads the host's slot tables to the device on st from the next pinned
// image; fault_expert >= 0 plants a wrong tag for that expert's slot.
static cudaError_t upload_tables(moe_residency* R, cudaStream_t st, int fault_expert) {
  const int i = R->tab_next;
  R->tab_next = (i + 1) % kTabRing;
  cudaError_t e;
  if (R->tab_used[i] && (e = cudaEventSynchronize(R->ev_tab[i]))) return e;
  int32_t* h = R->h_tab[i];
  std::memcpy(h, R->slot_of.data(), static_cast<size_t>(R->E) * 4);
  std::memcpy(h + R->E, R->slot_expert.data(), static_cast<size_t>(R->n_slots) * 4);
  if (fault_expert >= 0) h[R->E + R->slot_of[fault_expert]] = (fault_expert + 1) % R->E;
  if ((e = cudaMemcpyAsync(R->d_tables, h, static_cast<size_t>(R->E + R->n_slots) * 4,
                           cudaMemcpyHostToDevice, st)) ||
      (e = cudaEventRecord(R->ev_tab[i], st)))
    return e;
  R->tab_used[i] = true;
  return cudaSuccess;
}

extern "C" int moe_residency_decode(moe_residency* R, const uint16_t* x, int32_t B, uint16_t* out_bf16,
                                    float* out_f32, int32_t* ids, float* weights, void* workspace,
                                    size_t workspace_bytes, void* main_stream, void* copy_stream) {
  static const char* kName = "moe_residency_decode";
  if (!res_valid(R)) return moe::report_error(MOE_ERR_ARG, "moe_residency_decode: invalid residency handle");
  moe::LayerArgs a;
  bool single = false;
  int num_sms = 0;
  int rc = moe::prepare_cached_decode(R->layer, x, B, out_bf16, out_f32, ids, weights, workspace,
                                      workspace_bytes, R->pool, R->d_tables, R->d_tables + R->E,
                                      R->n_slots, &a, &single, &num_sms, kName);
  if (rc || B == 0) return rc;
  cudaStream_t M = static_cast<cudaStream_t>(main_stream), C = static_cast<cudaStream_t>(copy_stream);
  const size_t nid = static_cast<size_t>(B) * R->k;

  // 1. router, ids to the host, the shared expert's gate|up
  cudaError_t e = single ? moe::launch_b1_router(a, num_sms, M) : moe::launch_decode_router(a, num_sms, M);
  if (e) return moe::report_cuda(e, "moe_residency_decode: router");
  if ((e = cudaMemcpyAsync(R->h_ids, ids, nid * 4, cudaMemcpyDeviceToHost, M)) ||
      (e = cudaEventRecord(R->ev_ids, M)))
    return moe::report_cuda(e, "moe_residency_decode: ids to host");
  if (single && (e = moe::launch_b1_shared(a, num_sms, M)))
    return moe::report_cuda(e, "moe_residency_decode: shared expert");
  if ((e = cudaEventSynchronize(R->ev_ids))) return moe::report_cuda(e, "moe_residency_decode: wait for ids");

  // 2. the step's distinct experts (validated: the host never indexes with a
  // bad id), counted and pinned
  const int64_t step = R->step + 1;
  R->order.clear();
  for (size_t i = 0; i < nid; ++i) {
    const int32_t ex = R->h_ids[i];
    if (ex < 0 || ex >= R->E)
      return moe::report_error(MOE_ERR_RESIDENCY, "moe_residency_decode: the router returned an expert id out of range (see moe_check)");
    if (R->pinned_at[ex] != step) R->pinned_at[ex] = step, R->order.push_back(ex);
  }
  if (static_cast<int>(R->order.size()) > R->n_slots) {
    // more experts than slots: waves of consecutive tokens, each a step of
    // its own (its router runs again; a single token always fits)
    for (int32_t ex : R->order) R->pinned_at[ex] = R->step;  // leave the state as it was
    std::vector<int> starts;
    plan_waves(R, B, &starts);
    starts.push_back(B);
    const size_t H = moe::layer_desc(R->layer)->hidden, k = R->k;
    for (size_t w = 0; w + 1 < starts.size(); ++w) {
      const int t0 = starts[w], n = starts[w + 1] - t0;
      rc = moe_residency_decode(R, x + t0 * H, n, out_bf16 + t0 * H, out_f32 ? out_f32 + t0 * H : nullptr,
                                ids + t0 * k, weights + t0 * k, workspace, workspace_bytes, main_stream,
                                copy_stream);
      if (rc) return rc;
    }
    return MOE_OK;
  }
  // optional payload check of records about to be uploaded for the first
  // time; a mismatch refuses the step before any state changes
  if (!R->crc_expect.empty()) {
    for (int32_t ex : R->order) {
      if (R->slot_of[ex] >= 0 || R->crc_checked[ex]) continue;
      const uint32_t got = moe_crc32(R->host + static_cast<size_t>(ex) * R->stride, R->rec_bytes);
      if (got != R->crc_expect[ex]) {
        for (int32_t e2 : R->order) R->pinned_at[e2] = R->step;  // leave the state as it was
        char msg[160];
        std::snprintf(msg, sizeof msg,
                      "moe_residency_decode: host record of expert %d fails its CRC-32 check (0x%08x, expected 0x%08x)",
                      static_cast<int>(ex), got, R->crc_expect[ex]);
        return moe::report_error(MOE_ERR_RESIDENCY, msg);
      }
      R->crc_checked[ex] = 1;
    }
  }
  R->step = step;
  for (int32_t ex : R->order) R->count[ex] += 1, R->last_use[ex] = step;
  for (int32_t ex : R->ahead_list) R->ahead[ex] = 0;  // a lookahead's pins end at this step
  R->ahead_list.clear();

  // 3. misses: choose slots, copy records on the side stream, after the
  // previous step's routed kernels and the previous lookahead's copies (both
  // may have used other streams)
  if ((e = cudaStreamWaitEvent(C, R->ev_done, 0)) || (e = cudaStreamWaitEvent(C, R->ev_ahead, 0)))
    return moe::report_cuda(e, "moe_residency_decode: order the copies");
  const int fault = R->fault;
  bool fault_used = false;
  uint64_t hits = 0, misses = 0, evictions = 0, bytes = 0, ahead_hits = 0;
  for (int32_t ex : R->order) {
    if (R->slot_of[ex] >= 0) {
      ++hits;
      if (R->fresh[ex]) ++ahead_hits, R->fresh[ex] = 0;
      continue;
    }
    const int s = choose_slot(R, false);  // never -1: distinct experts <= slots
    const int old = R->slot_expert[s];
    if (old >= 0) R->slot_of[old] = -1, R->fresh[old] = 0, ++evictions;
    ++misses;
    if (fault == MOE_RESIDENCY_FAULT_COPY && !fault_used) {
      e = cudaErrorInvalidValue;  // host-side stand-in for a failed copy
      fault_used = true;
    } else {
      e = cudaMemcpyAsync(R->pool + static_cast<size_t>(s) * R->stride, R->host + static_cast<size_t>(ex) * R->stride,
                          R->rec_bytes, cudaMemcpyHostToDevice, C);
    }
    if (e) {
      // the slot's contents are unknown now: it holds nothing
      R->slot_expert[s] = -1;
      R->stats.steps += 1, R->stats.hits += hits, R->stats.misses += misses;
      R->stats.evictions += evictions, R->stats.bytes_h2d += bytes, R->stats.lookahead_hits += ahead_hits;
      if (fault_used) R->fault = MOE_RESIDENCY_FAULT_NONE;
      return moe::report_cuda(e, "moe_residency_decode: record copy");
    }
    R->slot_expert[s] = ex, R->slot_of[ex] = s;
    bytes += R->rec_bytes;
  }

  // 4. slot tables (one small copy behind the records), then the routed part
  int fault_expert = -1;
  if (fault == MOE_RESIDENCY_FAULT_TAG) {
    fault_expert = R->order[0];  // this step's tag for it no longer matches
    R->fault = MOE_RESIDENCY_FAULT_NONE;
  }
  if ((e = upload_tables(R, C, fault_expert)) || (e = cudaEventRecord(R->ev_copy, C)) ||
      (e = cudaStreamWaitEvent(M, R->ev_copy, 0)))
    return moe::report_cuda(e, "moe_residency_decode: slot tables");
  R->stats.steps += 1, R->stats.hits += hits, R->stats.misses += misses;
  R->stats.evictions += evictions, R->stats.bytes_h2d += bytes, R->stats.lookahead_hits += ahead_hits;
  e = single ? moe::launch_b1_routed(a, num_sms, M)
      : a.cbs ? moe::launch_rvq_experts(a, num_sms, M)  // residual-VQ records
              : moe::launch_decode_experts(a, num_sms, M);
  if (e || (e = cudaEventRecord(R->ev_done, M))) return moe::report_cuda(e, "moe_residency_decode: routed experts");
  return MOE_OK;
}

extern "C" int moe_residency_lookahead(moe_residency* R, const uint16_t* x, int32_t B, int32_t n_ahead,
                                       int32_t* ids, float* weights, void* workspace, size_t workspace_bytes,
                                       void* stream, void* copy_stream) {
  static const char* kName = "moe_residency_lookahead";
  if (!res_valid(R)) return moe::report_error(MOE_ERR_ARG, "moe_residency_lookahead: invalid residency handle");
  if (n_ahead < 0 || n_ahead > R->k)
    return moe::report_error(MOE_ERR_ARG, "moe_residency_lookahead: n_ahead outside [0, top_k]");
  moe::LayerArgs a;
  bool single = false;
  int num_sms = 0;
  int rc = moe::prepare_route(R->layer, x, B, ids, weights, workspace, workspace_bytes, &a, &single, &num_sms, kName);
  if (rc || B == 0 || n_ahead == 0) return rc;
  cudaStream_t S = static_cast<cudaStream_t>(stream), C = static_cast<cudaStream_t>(copy_stream);
  const size_t nid = static_cast<size_t>(B) * R->k;

  // 1. the predicted routing, to the host
  cudaError_t e = single ? moe::launch_b1_router(a, num_sms, S) : moe::launch_decode_router(a, num_sms, S);
  if (e) return moe::report_cuda(e, "moe_residency_lookahead: router");
  if ((e = cudaMemcpyAsync(R->h_pids, ids, nid * 4, cudaMemcpyDeviceToHost, S)) ||
      (e = cudaEventRecord(R->ev_pids, S)) || (e = cudaEventSynchronize(R->ev_pids)))
    return moe::report_cuda(e, "moe_residency_lookahead: predicted ids to host");

  // 2. visiting order (rank-major), validated and, with checksums on,
  // checked before any state changes
  R->pred.clear();
  for (int r = 0; r < n_ahead; ++r)
    for (int t = 0; t < B; ++t) {
      const int32_t ex = R->h_pids[static_cast<size_t>(t) * R->k + r];
      if (ex < 0 || ex >= R->E)
        return moe::report_error(MOE_ERR_RESIDENCY, "moe_residency_lookahead: the router returned an expert id out of range (see moe_check)");
      R->pred.push_back(ex);
    }
  if (!R->crc_expect.empty()) {
    for (int32_t ex : R->pred) {
      if (R->slot_of[ex] >= 0 || R->crc_checked[ex]) continue;
      const uint32_t got = moe_crc32(R->host + static_cast<size_t>(ex) * R->stride, R->rec_bytes);
      if (got != R->crc_expect[ex]) {
        char msg[160];
        std::snprintf(msg, sizeof msg,
                      "moe_residency_lookahead: host record of expert %d fails its CRC-32 check (0x%08x, expected 0x%08x)",
                      static_cast<int>(ex), got, R->crc_expect[ex]);
        return moe::report_error(MOE_ERR_RESIDENCY, msg);
      }
      R->crc_checked[ex] = 1;
    }
  }
  for (int32_t ex : R->pred)
    if (!R->ahead[ex]) R->ahead[ex] = 1, R->ahead_list.push_back(ex);

  // 3. copies, after the last step's kernels and the last lookahead
  if ((e = cudaStreamWaitEvent(C, R->ev_done, 0)) || (e = cudaStreamWaitEvent(C, R->ev_ahead, 0)))
    return moe::report_cuda(e, "moe_residency_lookahead: order the copies");
  uint64_t copies = 0, evictions = 0, bytes = 0;
  for (int32_t ex : R->pred) {
    if (R->slot_of[ex] >= 0) continue;  // resident (or copied by an earlier repeat)
    const int s = choose_slot(R, true);
    if (s < 0) continue;                // every slot pinned: dropped
    const int old = R->slot_expert[s];
    if (old >= 0) R->slot_of[old] = -1, R->fresh[old] = 0, ++evictions;
    if (R->fault == MOE_RESIDENCY_FAULT_COPY) {
      e = cudaErrorInvalidValue;  // host-side stand-in for a failed copy
      R->fault = MOE_RESIDENCY_FAULT_NONE;
    } else {
      e = cudaMemcpyAsync(R->pool + static_cast<size_t>(s) * R->stride, R->host + static_cast<size_t>(ex) * R->stride,
                          R->rec_bytes, cudaMemcpyHostToDevice, C);
    }
    if (e) {
      R->slot_expert[s] = -1;  // contents unknown: the slot holds nothing
      R->stats.lookaheads += 1, R->stats.lookahead_copies += copies;
      R->stats.evictions += evictions, R->stats.lookahead_bytes += bytes;
      if (copies) cudaEventRecord(R->ev_ahead, C);  // the next step still orders after the copies issued
      return moe::report_cuda(e, "moe_residency_lookahead: record copy");
    }
    R->slot_expert[s] = ex, R->slot_of[ex] = s, R->fresh[ex] = 1;
    ++copies, bytes += R->rec_bytes;
  }
  if (copies && ((e = upload_tables(R, C, -1)) || (e = cudaEventRecord(R->ev_ahead, C)))) {
    cudaEventRecord(R->ev_ahead, C);
    return moe::report_cuda(e, "moe_residency_lookahead: slot tables");
  }
  R->stats.lookaheads += 1, R->stats.lookahead_copies += copies;
  R->stats.evictions += evictions, R->stats.lookahead_bytes += bytes;
  return MOE_OK;
}

extern "C" int moe_residency_stats(const moe_residency* R, moe_residency_stats_t* out) {
  if (!res_valid(R) || !out) return moe::report_error(MOE_ERR_ARG, "moe_residency_stats: invalid arguments");
  *out = R->stats;
  return MOE_OK;
}

extern "C" int moe_residency_slots(const moe_residency* R, int32_t* slot_expert, int32_t n) {
  if (!res_valid(R) || !slot_expert || n < R->n_slots)
    return moe::report_error(MOE_ERR_ARG, "moe_residency_slots: invalid arguments (n must be >= n_slots)");
  for (int s = 0; s < R->n_slots; ++s) slot_expert[s] = R->slot_expert[s];
  return MOE_OK;
}

extern "C" int moe_residency_verify(moe_residency* R, const uint32_t* crc) {
  if (!res_valid(R)) return moe::report_error(MOE_ERR_ARG, "moe_residency_verify: invalid residency handle");
  if (!crc) {
    R->crc_expect.clear(), R->crc_checked.clear();
    return MOE_OK;
  }
  R->crc_expect.assign(crc, crc + R->E);
  R->crc_checked.assign(R->E, 0);
  // records already resident were uploaded unchecked: each is checked now
  for (int s = 0; s < R->n_slots; ++s) {
    const int ex = R->slot_expert[s];
    if (ex < 0) continue;
    if (moe_crc32(R->host + static_cast<size_t>(ex) * R->stride, R->rec_bytes) != R->crc_expect[ex]) {
      R->crc_expect.clear(), R->crc_checked.clear();
      return moe::report_error(MOE_ERR_RESIDENCY, "moe_residency_verify: a resident record fails its CRC-32 check");
    }
    R->crc_checked[ex] = 1;
  }
  return MOE_OK;
}

extern "C" int moe_residency_set_fault(moe_residency* R, int32_t mode) {
  if (!res_valid(R)) return moe::report_error(MOE_ERR_ARG, "moe_residency_set_fault: invalid residency handle");
  if (mode != MOE_RESIDENCY_FAULT_NONE && mode != MOE_RESIDENCY_FAULT_TAG && mode != MOE_RESIDENCY_FAULT_COPY)
    return moe::report_error(MOE_ERR_ARG, "moe_residency_set_fault: unknown mode");
  R->fault = mode;
  return MOE_OK;
}

static void destroy(moe_residency* R) {
  for (cudaEvent_t ev : {R->ev_ids, R->ev_copy, R->ev_pids, R->ev_done, R->ev_ahead})
    if (ev) cudaEventDestroy(ev);
  for (int i = 0; i < kTabRing; ++i) {
    if (R->ev_tab[i]) cudaEventDestroy(R->ev_tab[i]);
    if (R->h_tab[i]) cudaFreeHost(R->h_tab[i]);
  }
  if (R->h_ids) cudaFreeHost(R->h_ids);
  if (R->h_pids) cudaFreeHost(R->h_pids);
  R->magic = 0;
  delete R;
}

extern "C" void moe_residency_close(moe_residency* R) {
  if (res_valid(R)) destroy(R);
}
