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
// Optional payload check (WASTE page, section "Disk streaming mimarisi": a
// crc32 of each record, off by default, worth running once on records of
// uncertain origin): with moe_residency_verify, a record's CRC-32 is
// computed on the host before its first upload and compared with the
// caller's value; a mismatch refuses the step, cache state unchanged.
#include <cstdint>
#include <cstdio>
#include <cstring>
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
cudaError_t launch_b1_router(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_b1_shared(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_b1_routed(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_decode_router(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_decode_experts(const LayerArgs& a, int num_sms, cudaStream_t st);
}  // namespace moe

namespace {

constexpr uint32_t kResMagic = 0x52657331u;  // "Res1"

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
  int32_t* h_tables;          // pinned mirror uploaded each step
  int32_t* h_ids;             // pinned: the step's ids [max_tokens][k]
  cudaEvent_t ev_ids, ev_copy;
  // cache state (host)
  std::vector<int32_t> slot_expert;  // [n_slots] expert held, -1 = empty
  std::vector<int32_t> slot_of;      // [E] slot holding the expert, -1 = not resident
  std::vector<int64_t> count, last_use;
  std::vector<int64_t> pinned_at;    // [E] step that pinned the expert
  std::vector<int32_t> order;        // the step's distinct experts, first-appearance order
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
  R->order.reserve(static_cast<size_t>(R->max_tokens) * R->k);
  const size_t tb = static_cast<size_t>(R->E + n_slots) * 4;
  if ((e = cudaHostAlloc(&R->h_tables, tb, cudaHostAllocDefault)) ||
      (e = cudaHostAlloc(&R->h_ids, static_cast<size_t>(R->max_tokens) * R->k * 4, cudaHostAllocDefault)) ||
      (e = cudaEventCreateWithFlags(&R->ev_ids, cudaEventDisableTiming)) ||
      (e = cudaEventCreateWithFlags(&R->ev_copy, cudaEventDisableTiming))) {
    destroy(R);
    return moe::report_cuda(e, "moe_residency_open: pinned buffers / events");
  }
  for (int i = 0; i < R->E + n_slots; ++i) R->h_tables[i] = -1;
  if ((e = cudaMemcpy(R->d_tables, R->h_tables, tb, cudaMemcpyHostToDevice))) {
    destroy(R);
    return moe::report_cuda(e, "moe_residency_open: slot tables");
  }
  R->magic = kResMagic;
  *out = R;
  return MOE_OK;
}

// Victim slot for a miss: the lowest empty slot, else the unpinned resident
// with the lowest (count, last use, id); -1 if every slot is pinned.
static int choose_slot(const moe_residency* R) {
  int best = -1;
  for (int s = 0; s < R->n_slots; ++s) {
    const int e = R->slot_expert[s];
    if (e < 0) return s;
    if (R->pinned_at[e] == R->step) continue;
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
    for (int32_t ex : R->order) R->pinned_at[ex] = R->step;  // leave the state as it was
    return moe::report_error(MOE_ERR_RESIDENCY, "moe_residency_decode: the step needs more distinct experts than the cache has slots");
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

  // 3. misses: choose slots, copy records on the side stream
  const int fault = R->fault;
  bool fault_used = false;
  uint64_t hits = 0, misses = 0, evictions = 0, bytes = 0;
  for (int32_t ex : R->order) {
    if (R->slot_of[ex] >= 0) {
      ++hits;
      continue;
    }
    const int s = choose_slot(R);  // never -1: distinct experts <= slots
    const int old = R->slot_expert[s];
    if (old >= 0) R->slot_of[old] = -1, ++evictions;
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
      R->stats.evictions += evictions, R->stats.bytes_h2d += bytes;
      if (fault_used) R->fault = MOE_RESIDENCY_FAULT_NONE;
      return moe::report_cuda(e, "moe_residency_decode: record copy");
    }
    R->slot_expert[s] = ex, R->slot_of[ex] = s;
    bytes += R->rec_bytes;
  }

  // 4. slot tables (one small copy behind the records), then the routed part
  std::memcpy(R->h_tables, R->slot_of.data(), static_cast<size_t>(R->E) * 4);
  std::memcpy(R->h_tables + R->E, R->slot_expert.data(), static_cast<size_t>(R->n_slots) * 4);
  if (fault == MOE_RESIDENCY_FAULT_TAG) {
    const int32_t ex = R->order[0];
    R->h_tables[R->E + R->slot_of[ex]] = (ex + 1) % R->E;  // this step's tag no longer matches
    R->fault = MOE_RESIDENCY_FAULT_NONE;
  }
  if ((e = cudaMemcpyAsync(R->d_tables, R->h_tables, static_cast<size_t>(R->E + R->n_slots) * 4,
                           cudaMemcpyHostToDevice, C)) ||
      (e = cudaEventRecord(R->ev_copy, C)) || (e = cudaStreamWaitEvent(M, R->ev_copy, 0)))
    return moe::report_cuda(e, "moe_residency_decode: slot tables");
  R->stats.steps += 1, R->stats.hits += hits, R->stats.misses += misses;
  R->stats.evictions += evictions, R->stats.bytes_h2d += bytes;
  e = single ? moe::launch_b1_routed(a, num_sms, M) : moe::launch_decode_experts(a, num_sms, M);
  if (e) return moe::report_cuda(e, "moe_residency_decode: routed experts");
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
  if (R->ev_ids) cudaEventDestroy(R->ev_ids);
  if (R->ev_copy) cudaEventDestroy(R->ev_copy);
  if (R->h_tables) cudaFreeHost(R->h_tables);
  if (R->h_ids) cudaFreeHost(R->h_ids);
  R->magic = 0;
  delete R;
}

extern "C" void moe_residency_close(moe_residency* R) {
  if (res_valid(R)) destroy(R);
}
