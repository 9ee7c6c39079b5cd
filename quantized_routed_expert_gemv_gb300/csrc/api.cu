// api.cu -- the C ABI of include/moe.h: argument validation, layer
// geometry, workspace carving and kernel launch order.  No CPU compute path
// exists: every step of the layer runs in the kernels of decode.cu /
// prefill.cu.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "kernels.h"
#include "tma.cuh"

namespace moe {
size_t decode_smem_need(const LayerArgs& a, int num_sms);
size_t prefill_smem_need(const LayerArgs& a, int num_sms);
cudaError_t set_decode_attributes(int smem_optin);
cudaError_t set_b1_attributes(int smem_optin);
bool plan_b1(LayerArgs& a, int num_sms, int smem_optin);
cudaError_t launch_decode_b1(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_stage_x(const void* src, void* dst, size_t bytes, cudaStream_t st);
cudaError_t launch_decode(const LayerArgs& a, int num_sms, cudaStream_t st);
cudaError_t set_prefill_attributes(int smem_optin);
cudaError_t launch_prefill(const LayerArgs& a, const LayerMaps* maps, int num_sms, cudaStream_t st);
cudaError_t build_layer_maps(const LayerArgs& a, LayerMaps* out);
bool prefill_tc_ok(const LayerArgs& a, int T);
size_t prefill_workspace_bytes(const LayerArgs& a, int T);
size_t rvq_smem_need(const LayerArgs& a);
cudaError_t set_rvq_attributes(int smem_optin);
cudaError_t launch_decode_rvq(const LayerArgs& a, int num_sms, cudaStream_t st);
size_t rvq_partial_floats(int H, int k, int F, int Fs, int T, int which);
bool plan_bt(LayerArgs& a, int num_sms, int smem_optin);
cudaError_t set_bt_attributes(int smem_optin);
cudaError_t launch_decode_bt(const LayerArgs& a, int num_sms, cudaStream_t st);
}  // namespace moe

using moe::LayerArgs;
using moe::RecordOffsets;

static thread_local char g_err[512] = "no error";

static int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

static int cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

static constexpr uint32_t kMagic = 0x4D6F4531u;  // "MoE1"

struct moe_layer {
  uint32_t magic;
  moe_layer_desc d;
  moe_layer_weights w;
  RecordOffsets off_r, off_s;
  int device, num_sms, smem_optin;
  cudaEvent_t prof[4];
  int prof_on;
  moe::LayerMaps maps;  // tiled-load descriptors of the code matrices (prefill)
  // moe_decode_host: page-locked staging buffers for the inputs and the
  // outputs (allocated by the first call, sized for max_tokens, freed by
  // moe_close), a private stream and a few captured steps (copy in, kernels)
  // replayed as CUDA graphs.  The output buffer is mapped: the kernels write
  // the outputs, ids and weights straight into it (host_out_dev).
  std::mutex* host_mu;
  uint8_t* host_in;
  uint8_t* host_in_dev;
  uint8_t* host_out;
  uint8_t* host_out_dev;
  size_t host_out_bytes;
  cudaStream_t host_st;
  struct HostGraph {
    void* ws;
    int B, f32;
    cudaGraphExec_t exec;
  } hg[4];
  int hg_next;
};

static bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

static bool dim_ok(int v) { return v >= 64 && v <= moe::kMaxDim && v % 64 == 0; }

static RecordOffsets offsets_of(int H, int F) {
  RecordOffsets o;
  const uint64_t h = static_cast<uint64_t>(H), f = static_cast<uint64_t>(F);
  const uint64_t mc = f * h / 2, msb = f * (h / 64) * 4, dsb = h * (f / 64) * 4;
  o.gate_codes = 0;
  o.up_codes = mc;
  o.down_codes = 2 * mc;
  o.gate_sb = 3 * mc;
  o.up_sb = o.gate_sb + msb;
  o.down_sb = o.up_sb + msb;
  o.bytes = o.down_sb + dsb;
  o.stride = (o.bytes + 4095u) / 4096u * 4096u;
  return o;
}

// 3-bit residual VQ (wbits = 3): code bytes only, 3 per 8 weights.
static RecordOffsets rvq_offsets_of(int H, int F) {
  RecordOffsets o;
  const uint64_t mat = static_cast<uint64_t>(F) * static_cast<uint64_t>(H) / 8 * 3;
  o.gate_codes = 0;
  o.up_codes = mat;
  o.down_codes = 2 * mat;
  o.bytes = 3 * mat;
  o.gate_sb = o.up_sb = o.down_sb = o.bytes;
  o.stride = (o.bytes + 4095u) / 4096u * 4096u;
  return o;
}

static RecordOffsets offsets_for(int wbits, int H, int F) {
  return wbits == 3 ? rvq_offsets_of(H, F) : offsets_of(H, F);
}

static void copy_layout(const RecordOffsets& o, moe_record_layout* out) {
  out->gate_codes = o.gate_codes, out->up_codes = o.up_codes, out->down_codes = o.down_codes;
  out->gate_sb = o.gate_sb, out->up_sb = o.up_sb, out->down_sb = o.down_sb;
  out->bytes = o.bytes, out->stride = o.stride;
}

extern "C" int moe_rvq_record_layout_of(int32_t hidden, int32_t ffn, moe_record_layout* out) {
  if (!out) return fail(MOE_ERR_ARG, "moe_rvq_record_layout_of: out is NULL");
  if (!dim_ok(hidden) || !dim_ok(ffn))
    return fail(MOE_ERR_ARG, "moe_rvq_record_layout_of: hidden=%d ffn=%d must be multiples of 64 in [64, %d]",
                hidden, ffn, moe::kMaxDim);
  copy_layout(rvq_offsets_of(hidden, ffn), out);
  return MOE_OK;
}

extern "C" int moe_record_layout_of(int32_t hidden, int32_t ffn, moe_record_layout* out) {
  if (!out) return fail(MOE_ERR_ARG, "moe_record_layout_of: out is NULL");
  if (!dim_ok(hidden) || !dim_ok(ffn))
    return fail(MOE_ERR_ARG, "moe_record_layout_of: hidden=%d ffn=%d must be multiples of 64 in [64, %d]",
                hidden, ffn, moe::kMaxDim);
  copy_layout(offsets_of(hidden, ffn), out);
  return MOE_OK;
}

static int check_desc(const moe_layer_desc* d) {
  if (!d) return fail(MOE_ERR_ARG, "desc is NULL");
  if (!dim_ok(d->hidden)) return fail(MOE_ERR_ARG, "hidden=%d: must be a multiple of 64 in [64, %d]", d->hidden, moe::kMaxDim);
  if (d->n_experts < 1 || d->n_experts > moe::kMaxExperts)
    return fail(MOE_ERR_ARG, "n_experts=%d: must be in [1, %d]", d->n_experts, moe::kMaxExperts);
  if (d->top_k < 1 || d->top_k > std::min(d->n_experts, moe::kMaxTopK))
    return fail(MOE_ERR_ARG, "top_k=%d: must be in [1, min(n_experts, %d)]", d->top_k, moe::kMaxTopK);
  if (!dim_ok(d->ffn)) return fail(MOE_ERR_ARG, "ffn=%d: must be a multiple of 64 in [64, %d]", d->ffn, moe::kMaxDim);
  if (d->shared_ffn != 0 && !dim_ok(d->shared_ffn))
    return fail(MOE_ERR_ARG, "shared_ffn=%d: must be 0 or a multiple of 64 in [64, %d]", d->shared_ffn, moe::kMaxDim);
  if (d->group != 64) return fail(MOE_ERR_ARG, "group=%d: only 64 is supported", d->group);
  if (d->wbits != 4 && d->wbits != 3)
    return fail(MOE_ERR_ARG, "wbits=%d: 4 (affine, group 64) or 3 (residual VQ) are supported", d->wbits);
  if (d->rbits != 8) return fail(MOE_ERR_ARG, "rbits=%d: only 8 is supported", d->rbits);
  if (d->max_tokens < 1 || d->max_tokens > moe::kMaxTokens)
    return fail(MOE_ERR_ARG, "max_tokens=%d: must be in [1, %d]", d->max_tokens, moe::kMaxTokens);
  return MOE_OK;
}

extern "C" size_t moe_expert_bytes(const moe_layer_desc* desc, int32_t ffn) {
  if (!desc || !dim_ok(desc->hidden) || !dim_ok(ffn)) return 0;
  return static_cast<size_t>(offsets_for(desc->wbits, desc->hidden, ffn).stride);
}

static LayerArgs base_args(const moe_layer* L) {
  LayerArgs a;
  std::memset(&a, 0, sizeof a);
  a.H = L->d.hidden, a.E = L->d.n_experts, a.k = L->d.top_k, a.F = L->d.ffn, a.Fs = L->d.shared_ffn;
  a.records = static_cast<const uint8_t*>(L->w.expert_records);
  a.shared = static_cast<const uint8_t*>(L->w.shared_record);
  a.rcodes = L->w.router_codes;
  a.rsb = L->w.router_sb;
  a.beta = L->w.router_logit_bias;
  a.cbs = L->d.wbits == 3 ? L->w.expert_codebooks : nullptr;
  a.off_r = L->off_r, a.off_s = L->off_s;
  a.prof_on = L->prof_on;
  for (int i = 0; i < 4; ++i) a.prof[i] = L->prof_on ? static_cast<void*>(L->prof[i]) : nullptr;
  return a;
}

extern "C" int moe_open(const moe_layer_desc* desc, const moe_layer_weights* w, moe_layer** out) {
  if (!out) return fail(MOE_ERR_ARG, "moe_open: out is NULL");
  *out = nullptr;
  int rc = check_desc(desc);
  if (rc) return rc;
  if (!w) return fail(MOE_ERR_ARG, "moe_open: weights is NULL");
  if (!w->router_codes || !w->router_sb) return fail(MOE_ERR_ARG, "moe_open: router_codes/router_sb are NULL");
  if ((desc->shared_ffn > 0) != (w->shared_record != nullptr))
    return fail(MOE_ERR_ARG, "moe_open: shared_record must be non-NULL exactly when shared_ffn > 0");
  if (!aligned(w->router_codes, 16) || !aligned(w->router_sb, 16) ||
      !aligned(w->router_logit_bias, 16))
    return fail(MOE_ERR_ALIGN, "moe_open: router pointers must be 16-byte aligned");
  if (!aligned(w->expert_records, 256) || !aligned(w->shared_record, 256))
    return fail(MOE_ERR_ALIGN, "moe_open: expert records must be 256-byte aligned");
  if (desc->wbits == 3 && !w->expert_codebooks)
    return fail(MOE_ERR_ARG, "moe_open: wbits=3 needs expert_codebooks");
  if (!aligned(w->expert_codebooks, 16))
    return fail(MOE_ERR_ALIGN, "moe_open: expert_codebooks must be 16-byte aligned");

  moe_layer* L = new (std::nothrow) moe_layer;
  if (!L) return fail(MOE_ERR_NOMEM, "moe_open: out of host memory");
  std::memset(L, 0, sizeof *L);
  L->magic = kMagic;
  L->d = *desc;
  L->w = *w;
  const int H = desc->hidden, F = desc->ffn, Fs = desc->shared_ffn;
  L->off_r = offsets_for(desc->wbits, H, F);
  L->off_s = Fs ? offsets_for(desc->wbits, H, Fs) : RecordOffsets{};

  cudaError_t e = cudaGetDevice(&L->device);
  if (e) {
    delete L;
    return cuda_fail(e, "moe_open: cudaGetDevice");
  }
  int major = 0, minor = 0, smem_optin = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, L->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, L->device);
  cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device);
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, L->device);
  L->smem_optin = smem_optin;
  if (major != 10 || minor != 3) {
    const int dev = L->device;
    delete L;
    return fail(MOE_ERR_UNSUPPORTED, "moe_open: device %d is sm_%d%d; this library is built for sm_103a",
                dev, major, minor);
  }
  const LayerArgs a = base_args(L);
  const bool rvq = desc->wbits == 3;
  const size_t need = rvq ? moe::rvq_smem_need(a)
                          : std::max(moe::decode_smem_need(a, L->num_sms), moe::prefill_smem_need(a, L->num_sms));
  if (need + 1024 > static_cast<size_t>(smem_optin)) {
    delete L;
    return fail(MOE_ERR_UNSUPPORTED, "moe_open: kernels need %zu B of shared memory, device allows %d",
                need, smem_optin);
  }
  if ((e = moe::set_decode_attributes(smem_optin)) || (e = moe::set_b1_attributes(smem_optin)) ||
      (e = moe::set_prefill_attributes(smem_optin)) || (e = moe::set_rvq_attributes(smem_optin)) ||
      (e = moe::set_bt_attributes(smem_optin))) {
    delete L;
    return cuda_fail(e, "moe_open: cudaFuncSetAttribute");
  }
  if (!rvq && (e = moe::build_layer_maps(a, &L->maps))) {
    delete L;
    return cuda_fail(e, "moe_open: tensor maps of the code matrices");
  }
  L->host_mu = new (std::nothrow) std::mutex;
  if (!L->host_mu) {
    delete L;
    return fail(MOE_ERR_NOMEM, "moe_open: out of host memory");
  }
  *out = L;
  return MOE_OK;
}

extern "C" void moe_close(moe_layer* L) {
  if (L && L->magic == kMagic) {
    L->magic = 0;
    for (auto& g : L->hg)
      if (g.exec) cudaGraphExecDestroy(g.exec);
    if (L->host_st) cudaStreamDestroy(L->host_st);
    if (L->host_in) cudaFreeHost(L->host_in);
    if (L->host_out) cudaFreeHost(L->host_out);
    delete L->host_mu;
    delete L;
  }
}

// ---- workspace -------------------------------------------------------------
// [control: 64 words][entry counters][row-tile counters][fixed-point h]
// [down partial outputs][logits][grouping][h][h_shared][host-entry staging]
// [prefill scratch].  The control block and the counters persist between
// calls (kept at zero by the kernels, cleared by moe_check after a device
// error); everything after them is per-call scratch.

// The persistent control block: 64 control words, per-entry h counters (the
// shared expert and up to kMaxExperts routed experts), per down row tile
// counters (at most H / 8 tiles), each region rounded to 256 bytes.
constexpr size_t round256(size_t v) { return (v + 255) / 256 * 256; }
constexpr size_t kCtlBytes = round256(64 * 4);
constexpr size_t kHcntBytes = round256((moe::kMaxExperts + 1) * 4);
constexpr size_t kTcntBytes = round256(moe::kMaxDim / 8 * 4);
// Bytes at the start of a workspace that persist between calls.
constexpr size_t kPersistentBytes = kCtlBytes + kHcntBytes + kTcntBytes;

struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  }
};

static size_t carve(const moe_layer* L, int T, moe::Workspace* ws, uint8_t* base,
                    size_t* prefill_off) {
  const size_t H = L->d.hidden, E = L->d.n_experts, k = L->d.top_k, F = L->d.ffn,
               Fs = L->d.shared_ffn, t = static_cast<size_t>(T);
  Carve c;
  const bool rvq = L->d.wbits == 3;
  const size_t o_ctl = c.take(kCtlBytes), o_hcnt = c.take(kHcntBytes), o_tcnt = c.take(kTcntBytes);
  // Fixed-point h of the fused kernels, per 32-value chunk 64 bytes of words
  // and 4 group scales and sums (96 B): one token, a block per expert entry
  // (k routed rows of F, the shared row of Fs); few tokens, a block per
  // (expert, token) pair padded to 128-byte lines.  The few-token buffers are sized for
  // min(T, kBtMaxTokens) tokens, so a workspace for T serves every smaller
  // batch.
  const size_t tb = rvq ? 0 : std::min(t, static_cast<size_t>(moe::kBtMaxTokens));
  const auto line128 = [](size_t v) { return (v + 127) / 128 * 128; };
  const size_t o_hx = c.take(std::max((k * (F / 32) + Fs / 32) * 96, tb * (k * line128(3 * F) + line128(3 * Fs))));
  const size_t o_yp = c.take(std::max(k + 1, tb * (k + (Fs ? 1 : 0))) * H * 4);
  const size_t o_xq = c.take(tb * (H / 32) * 72);
  const size_t o_log = c.take(t * E * 4);
  const size_t o_nact = c.take(16);
  const size_t o_ae = c.take(E * 4), o_ao = c.take(E * 4), o_ac = c.take(E * 4);
  const size_t o_pt = c.take(t * k * 4), o_ps = c.take(t * k * 4);
  const size_t o_h = c.take(t * k * F * 4), o_hs = c.take(t * Fs * 4);
  // host-entry staging: x, then the outputs back to back (bf16, ids,
  // weights, then f32).  The same offsets lay out the layer's mapped output
  // buffer, which the kernels write; the ids and weights here are the device
  // copies the expert kernels read.
  const size_t o_xs = c.take(t * H * 2), o_obs = c.take(t * H * 2);
  const size_t o_ids = c.take(t * k * 4), o_w = c.take(t * k * 4), o_ofs = c.take(t * H * 4);
  LayerArgs a = base_args(L);
  // residual-VQ layers: per-slice partial sums of every token (slices of 256 inputs)
  const size_t o_rg = c.take(rvq ? moe::rvq_partial_floats(H, k, F, Fs, T, 0) * 4 : 0);
  const size_t o_ru = c.take(rvq ? moe::rvq_partial_floats(H, k, F, Fs, T, 1) * 4 : 0);
  const size_t o_ry = c.take(rvq ? moe::rvq_partial_floats(H, k, F, Fs, T, 2) * 4 : 0);
  const size_t o_pf = c.take(rvq ? 0 : moe::prefill_workspace_bytes(a, T));
  if (ws && base) {
    ws->ctl = reinterpret_cast<unsigned*>(base + o_ctl);
    ws->hcnt = reinterpret_cast<unsigned*>(base + o_hcnt);
    ws->tcnt = reinterpret_cast<unsigned*>(base + o_tcnt);
    ws->ypart = reinterpret_cast<float*>(base + o_yp);
    ws->xq = base + o_xq;
    ws->hx = base + o_hx;
    ws->logits = reinterpret_cast<float*>(base + o_log);
    ws->n_act = reinterpret_cast<int*>(base + o_nact);
    ws->act_expert = reinterpret_cast<int*>(base + o_ae);
    ws->act_off = reinterpret_cast<int*>(base + o_ao);
    ws->act_cnt = reinterpret_cast<int*>(base + o_ac);
    ws->pair_token = reinterpret_cast<int*>(base + o_pt);
    ws->pair_slot = reinterpret_cast<int*>(base + o_ps);
    ws->h = reinterpret_cast<float*>(base + o_h);
    ws->h_shared = reinterpret_cast<float*>(base + o_hs);
    ws->x_stage = reinterpret_cast<uint16_t*>(base + o_xs);
    ws->ob_stage = reinterpret_cast<uint16_t*>(base + o_obs);
    ws->of_stage = reinterpret_cast<float*>(base + o_ofs);
    ws->ids_stage = reinterpret_cast<int32_t*>(base + o_ids);
    ws->w_stage = reinterpret_cast<float*>(base + o_w);
    ws->rvq_g = rvq ? reinterpret_cast<float*>(base + o_rg) : nullptr;
    ws->rvq_u = rvq ? reinterpret_cast<float*>(base + o_ru) : nullptr;
    ws->rvq_y = rvq ? reinterpret_cast<float*>(base + o_ry) : nullptr;
  }
  if (prefill_off) *prefill_off = o_pf;
  if (ws && base) ws->pf = !rvq && moe::prefill_workspace_bytes(a, T) ? base + o_pf : nullptr;
  return c.off;
}

static bool valid(const moe_layer* L) { return L && L->magic == kMagic; }

extern "C" size_t moe_workspace_bytes(const moe_layer* L, int32_t max_tokens) {
  if (!valid(L) || max_tokens < 1 || max_tokens > L->d.max_tokens) return 0;
  return carve(L, max_tokens, nullptr, nullptr, nullptr);
}

extern "C" int moe_workspace_init(const moe_layer* L, void* ws, size_t bytes, void* stream) {
  if (!valid(L)) return fail(MOE_ERR_ARG, "moe_workspace_init: invalid layer handle");
  if (!ws) return fail(MOE_ERR_ARG, "moe_workspace_init: workspace is NULL");
  if (!aligned(ws, 256)) return fail(MOE_ERR_ALIGN, "moe_workspace_init: workspace must be 256-byte aligned");
  cudaError_t e = cudaMemsetAsync(ws, 0, bytes, static_cast<cudaStream_t>(stream));
  return e ? cuda_fail(e, "moe_workspace_init: cudaMemsetAsync") : MOE_OK;
}

enum class Path { kDecode, kPrefill, kRoute };  // kRoute: the router alone, no layer output

// Validates one call and fills `a` (geometry and workspace; the records are
// the layer's own unless the caller replaces them).  T == 0 is valid and
// leaves *a untouched.
static int prepare(moe_layer* L, const uint16_t* x, int32_t T, uint16_t* ob, float* of, int32_t* ids,
                   float* wts, void* ws, size_t ws_bytes, Path path, bool need_records, LayerArgs* a,
                   const char* name) {
  if (!valid(L)) return fail(MOE_ERR_ARG, "%s: invalid layer handle", name);
  const int cap = path == Path::kPrefill ? std::min(128, (int)L->d.max_tokens) : (int)L->d.max_tokens;
  if (T < 0 || T > cap) return fail(MOE_ERR_ARG, "%s: token count %d outside [0, %d]", name, T, cap);
  if (T == 0) return MOE_OK;
  if (!x || (!ob && path != Path::kRoute) || !ids || !wts || !ws)
    return fail(MOE_ERR_ARG, "%s: a required pointer is NULL", name);
  if (!aligned(x, 16) || !aligned(ob, 16) || !aligned(of, 16) || !aligned(ids, 16) || !aligned(wts, 16))
    return fail(MOE_ERR_ALIGN, "%s: activation/output pointers must be 16-byte aligned", name);
  if (!aligned(ws, 256)) return fail(MOE_ERR_ALIGN, "%s: workspace must be 256-byte aligned", name);
  if (need_records && !L->w.expert_records)
    return fail(MOE_ERR_ARG, "%s: layer has no resident expert records", name);
  size_t pf_off = 0;
  *a = base_args(L);
  const size_t need = carve(L, T, &a->ws, static_cast<uint8_t*>(ws), &pf_off);
  if (ws_bytes < need) return fail(MOE_ERR_ARG, "%s: workspace of %zu B is smaller than the %zu B needed", name, ws_bytes, need);
  a->T = T, a->x = x, a->out_bf16 = ob, a->out_f32 = of, a->ids = ids, a->weights = wts;
  (void)pf_off;
  return MOE_OK;
}

// Decode batches with B * top_k <= E (with uniform routing fewer than ~40%
// of the pairs repeat an expert) run one single-token pass per token: the
// single-token kernels stream weights several times faster than the grouped
// ones, which outweighs the repeated reads.  Measured at H=7168, E=512,
// top-16: B=32 per token 2.9 ms vs 4.3 ms on the tensor-core kernels.
static bool per_token_decode(const moe_layer* L, int T) {
  return T > 1 && T <= 64 && static_cast<long>(T) * L->d.top_k <= L->d.n_experts;
}

// Batches of 2..kBtMaxTokens tokens run the few-token fused kernel
// (decode_bt.cu): the single-token weight stream with a token loop per item.
static bool few_token_decode(const moe_layer* L, int T) {
  return T >= 2 && T <= moe::kBtMaxTokens && L->d.wbits == 4;
}

// plan_bt on a copy of `a`'s geometry fields (the single-token plan must
// hold too: the few-token kernel uses its row-lane mapping).
static bool bt_planned(const moe_layer* L, LayerArgs& a) {
  LayerArgs b = a;
  if (!moe::plan_b1(b, L->num_sms, L->smem_optin)) return false;
  if (!moe::plan_bt(b, L->num_sms, L->smem_optin)) return false;
  a = b;
  return true;
}

// ids_host / w_host: optional copies of ids and weights in mapped host
// memory, written by the router beside the device ones.  x_pdl: x is being
// written by the kernel launched just before this call (the host entry's
// staging kernel), which a single-token router may overlap.
static int run(moe_layer* L, const uint16_t* x, int32_t T, uint16_t* ob, float* of, int32_t* ids,
               float* wts, void* ws, size_t ws_bytes, void* stream, Path path, const char* name,
               int32_t* ids_host = nullptr, float* w_host = nullptr, bool x_pdl = false) {
  LayerArgs a;
  const int rc = prepare(L, x, T, ob, of, ids, wts, ws, ws_bytes, path, true, &a, name);
  if (rc || T == 0) return rc;
  a.ids_host = ids_host, a.weights_host = ids_host ? w_host : nullptr;
  a.x_pdl = x_pdl ? 1 : 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (L->d.wbits == 3) {
    // residual-VQ experts: their own decode kernels, any B; no chunked prefill
    if (path == Path::kPrefill) return fail(MOE_ERR_ARG, "%s: prefill chunks need wbits=4 experts", name);
    e = moe::launch_decode_rvq(a, L->num_sms, st);
  } else if (path == Path::kPrefill) {
    e = moe::launch_prefill(a, &L->maps, L->num_sms, st);
  } else if (T == 1 && moe::plan_b1(a, L->num_sms, L->smem_optin)) {
    e = moe::launch_decode_b1(a, L->num_sms, st);
  } else if (few_token_decode(L, T) && bt_planned(L, a)) {
    // A few tokens: one pass over the step's experts, each expert's weights
    // read once and applied to all of its tokens.
    e = moe::launch_decode_bt(a, L->num_sms, st);
  } else if (per_token_decode(L, T) && moe::plan_b1(a, L->num_sms, L->smem_optin)) {
    // Few tokens over many experts: the tokens share almost no expert, so a
    // grouped pass reads nearly the same weight bytes as one single-token
    // pass per token, and the single-token kernels stream them faster.
    e = cudaSuccess;
    for (int t = 0; t < T && e == cudaSuccess; ++t) {
      LayerArgs b = a;
      const size_t H = L->d.hidden, k = L->d.top_k;
      b.T = 1, b.x = x + t * H, b.out_bf16 = ob + t * H, b.out_f32 = of ? of + t * H : nullptr;
      b.ids = ids + t * k, b.weights = wts + t * k;
      if (ids_host) b.ids_host = ids_host + t * k, b.weights_host = w_host + t * k;
      b.x_pdl = t == 0 ? a.x_pdl : 0;  // later tokens follow the previous token's kernels
      b.prof_on = t == 0 ? a.prof_on : 0;  // the profiling hook times the first token's kernels
      e = moe::launch_decode_b1(b, L->num_sms, st);
    }
  } else if (moe::prefill_tc_ok(a, T) && L->maps.valid) {
    // Larger batches: the tensor-core kernels of the prefill chunk compute
    // the same layer with each expert's weights read once for all its tokens.
    e = moe::launch_prefill(a, &L->maps, L->num_sms, st);
  } else {
    e = moe::launch_decode(a, L->num_sms, st);
  }
  if (e) return cuda_fail(e, name);
  return MOE_OK;
}

extern "C" int moe_decode(moe_layer* L, const uint16_t* x, int32_t B, uint16_t* out_bf16, float* out_f32,
                          int32_t* ids, float* weights, void* ws, size_t ws_bytes, void* stream) {
  return run(L, x, B, out_bf16, out_f32, ids, weights, ws, ws_bytes, stream, Path::kDecode, "moe_decode");
}

extern "C" int moe_prefill_chunk(moe_layer* L, const uint16_t* x, int32_t T, uint16_t* out_bf16,
                                 float* out_f32, int32_t* ids, float* weights, void* ws, size_t ws_bytes,
                                 void* stream) {
  return run(L, x, T, out_bf16, out_f32, ids, weights, ws, ws_bytes, stream, Path::kPrefill,
             "moe_prefill_chunk");
}

// moe_decode_host's staging buffers and private stream, made once per layer.
static int host_entry_setup(moe_layer* L, void* ws) {
  if (L->host_out) return MOE_OK;
  const size_t H = L->d.hidden, n = static_cast<size_t>(L->d.max_tokens);
  moe::Workspace wm;
  carve(L, L->d.max_tokens, &wm, static_cast<uint8_t*>(ws), nullptr);
  const size_t out_bytes =
      static_cast<size_t>(reinterpret_cast<uint8_t*>(wm.of_stage) - reinterpret_cast<uint8_t*>(wm.ob_stage)) +
      n * H * 4;
  void *pin = nullptr, *pout = nullptr;
  cudaError_t e;
  if ((e = cudaHostAlloc(&pin, n * H * 2, cudaHostAllocMapped)))
    return cuda_fail(e, "moe_decode_host: page-locked input buffer");
  if ((e = cudaHostAlloc(&pout, out_bytes, cudaHostAllocMapped))) {
    cudaFreeHost(pin);
    return cuda_fail(e, "moe_decode_host: page-locked output buffer");
  }
  void *pin_dev = nullptr, *pout_dev = nullptr;
  if ((e = cudaHostGetDevicePointer(&pin_dev, pin, 0)) || (e = cudaHostGetDevicePointer(&pout_dev, pout, 0))) {
    cudaFreeHost(pin), cudaFreeHost(pout);
    return cuda_fail(e, "moe_decode_host: device address of a page-locked buffer");
  }
  if ((e = cudaStreamCreateWithFlags(&L->host_st, cudaStreamNonBlocking))) {
    cudaFreeHost(pin), cudaFreeHost(pout);
    L->host_st = nullptr;
    return cuda_fail(e, "moe_decode_host: capture stream");
  }
  L->host_in = static_cast<uint8_t*>(pin), L->host_out = static_cast<uint8_t*>(pout), L->host_out_bytes = out_bytes;
  L->host_out_dev = static_cast<uint8_t*>(pout_dev);
  L->host_in_dev = static_cast<uint8_t*>(pin_dev);
  return MOE_OK;
}

// Copy in, then the step, on `st`.  A small kernel copies x from the mapped
// input buffer into the workspace; a single-token router is launched as its
// programmatic dependent, so the router's launch and weight loads overlap the
// copy (other paths follow it in plain stream order).  The outputs land in
// the layer's mapped output buffer, at the offsets the workspace's output
// staging area has: the kernels write the bf16 (and f32) outputs there, and
// the router writes ids and weights both to the workspace (which the expert
// kernels read) and there.  No copy out: the host reads the buffer after the
// synchronisation.
static int host_entry_step(moe_layer* L, int32_t B, bool f32, const moe::Workspace& w, void* ws, size_t ws_bytes,
                           size_t o_ids, size_t o_w, size_t o_f, cudaStream_t st) {
  const size_t H = L->d.hidden;
  cudaError_t e = moe::launch_stage_x(L->host_in_dev, w.x_stage, static_cast<size_t>(B) * H * 2, st);
  if (e) return cuda_fail(e, "moe_decode_host: copy in");
  uint8_t* const hd = L->host_out_dev;
  return run(L, w.x_stage, B, reinterpret_cast<uint16_t*>(hd), f32 ? reinterpret_cast<float*>(hd + o_f) : nullptr,
             w.ids_stage, w.w_stage, ws, ws_bytes, st, Path::kDecode, "moe_decode_host",
             reinterpret_cast<int32_t*>(hd + o_ids), reinterpret_cast<float*>(hd + o_w), true);
}

extern "C" int moe_decode_host(moe_layer* L, const uint16_t* x_host, int32_t B, uint16_t* ob_host,
                               float* of_host, int32_t* ids_host, float* w_host, void* ws,
                               size_t ws_bytes, void* stream) {
  if (!valid(L)) return fail(MOE_ERR_ARG, "moe_decode_host: invalid layer handle");
  if (B < 0 || B > L->d.max_tokens) return fail(MOE_ERR_ARG, "moe_decode_host: B=%d outside [0, %d]", B, L->d.max_tokens);
  if (B == 0) return MOE_OK;
  if (!x_host || !ob_host || !ids_host || !w_host || !ws)
    return fail(MOE_ERR_ARG, "moe_decode_host: a required pointer is NULL");
  if (!aligned(ws, 256)) return fail(MOE_ERR_ALIGN, "moe_decode_host: workspace must be 256-byte aligned");
  moe::Workspace w;
  const size_t need = carve(L, B, &w, static_cast<uint8_t*>(ws), nullptr);
  if (ws_bytes < need) return fail(MOE_ERR_ARG, "moe_decode_host: workspace too small (%zu < %zu)", ws_bytes, need);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t H = L->d.hidden, k = L->d.top_k, b = static_cast<size_t>(B);
  // The staging area holds bf16 out, ids, weights and f32 out back to back:
  // one copy of [ob_stage, end) brings every requested output to the
  // layer's page-locked buffer, from which they are handed out.
  uint8_t* const s0 = reinterpret_cast<uint8_t*>(w.ob_stage);
  const size_t o_ids = reinterpret_cast<uint8_t*>(w.ids_stage) - s0;
  const size_t o_w = reinterpret_cast<uint8_t*>(w.w_stage) - s0;
  const size_t o_f = reinterpret_cast<uint8_t*>(w.of_stage) - s0;
  const bool f32 = of_host != nullptr;
  std::lock_guard<std::mutex> lock(*L->host_mu);
  int rc = host_entry_setup(L, ws);
  if (rc) return rc;
  std::memcpy(L->host_in, x_host, b * H * 2);
  // A step already captured for this workspace, batch and output set is
  // replayed as one graph launch; otherwise the step runs as plain launches
  // and is captured for the next call (every kernel has launched once by
  // then).  The profiling hook always takes plain launches.
  cudaGraphExec_t exec = nullptr;
  if (!L->prof_on)
    for (const auto& g : L->hg)
      if (g.exec && g.ws == ws && g.B == B && g.f32 == (f32 ? 1 : 0)) exec = g.exec;
  cudaError_t e;
  if (exec) {
    if ((e = cudaGraphLaunch(exec, st))) return cuda_fail(e, "moe_decode_host: graph launch");
  } else {
    if ((rc = host_entry_step(L, B, f32, w, ws, ws_bytes, o_ids, o_w, o_f, st))) return rc;
  }
  if ((e = cudaStreamSynchronize(st))) return cuda_fail(e, "moe_decode_host: synchronize");
  std::memcpy(ob_host, L->host_out, b * H * 2);
  std::memcpy(ids_host, L->host_out + o_ids, b * k * 4);
  std::memcpy(w_host, L->host_out + o_w, b * k * 4);
  if (f32) std::memcpy(of_host, L->host_out + o_f, b * H * 4);
  if (!exec && !L->prof_on) {
    // capture this step on the private stream; a failed capture only means
    // later calls keep the plain launches
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t ge = nullptr;
    if (cudaStreamBeginCapture(L->host_st, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
      const int crc = host_entry_step(L, B, f32, w, ws, ws_bytes, o_ids, o_w, o_f, L->host_st);
      const cudaError_t ce = cudaStreamEndCapture(L->host_st, &graph);
      if (crc == MOE_OK && ce == cudaSuccess && graph && cudaGraphInstantiate(&ge, graph, 0) == cudaSuccess) {
        auto& slot = L->hg[L->hg_next];
        if (slot.exec) cudaGraphExecDestroy(slot.exec);
        slot.ws = ws, slot.B = B, slot.f32 = f32 ? 1 : 0, slot.exec = ge;
        L->hg_next = (L->hg_next + 1) % 4;
      }
      if (graph) cudaGraphDestroy(graph);
    }
    cudaGetLastError();  // a capture that failed leaves no sticky error behind
  }
  return MOE_OK;
}

extern "C" int32_t moe_decode_kernels(const moe_layer* L, int32_t B) {
  if (!valid(L) || B < 0 || B > L->d.max_tokens) return -1;
  if (B == 0) return 0;
  if (L->d.wbits == 3) return 4;  // router, gate|up, down, combine for every token at once
  LayerArgs a = base_args(L);
  a.T = B;
  const int b1 = moe::plan_b1(a, L->num_sms, L->smem_optin) ? (a.f1_nst > 0 ? 2 : 3) : 0;
  if (B == 1 && b1) return b1;
  if (few_token_decode(L, B) && bt_planned(L, a)) return 3;
  if (per_token_decode(L, B) && b1) return B * b1;
  if (moe::prefill_tc_ok(a, B) && L->maps.valid) return 5;
  return 3;
}

// Reads the error word that device code latches at the start of workspace
// `ws` after synchronising `st`; after an error, zeroes the persistent block.
static int check_workspace(void* ws, cudaStream_t st, const char* name) {
  cudaError_t e = cudaStreamSynchronize(st);
  if (e) return cuda_fail(e, name);
  unsigned bits = 0;
  if ((e = cudaMemcpy(&bits, ws, 4, cudaMemcpyDeviceToHost))) return cuda_fail(e, name);
  if (bits == 0) return MOE_OK;
  // a step that gave up may leave claim and completion counters mid-count:
  // the whole persistent block goes back to zero with the error word
  if ((e = cudaMemset(ws, 0, kPersistentBytes))) return cuda_fail(e, name);
  if (bits & moe::kErrTimeout) return fail(MOE_ERR_TIMEOUT, "device code gave up a bounded wait (bits 0x%x)", bits);
  if (bits & moe::kErrResidency) return fail(MOE_ERR_RESIDENCY, "an expert slot did not hold the routed expert (bits 0x%x)", bits);
  return fail(MOE_ERR_ARG, "device code clamped an out-of-range routing value (bits 0x%x)", bits);
}

extern "C" int moe_check(const moe_layer* L, void* ws, void* stream) {
  if (!valid(L)) return fail(MOE_ERR_ARG, "moe_check: invalid layer handle");
  if (!ws) return fail(MOE_ERR_ARG, "moe_check: workspace is NULL");
  return check_workspace(ws, static_cast<cudaStream_t>(stream), "moe_check");
}

extern "C" int moe_set_profile_events(moe_layer* L, void* const* events) {
  if (!valid(L)) return fail(MOE_ERR_ARG, "moe_set_profile_events: invalid layer handle");
  if (!events) {
    L->prof_on = 0;
    return MOE_OK;
  }
  for (int i = 0; i < 4; ++i) {
    if (!events[i]) return fail(MOE_ERR_ARG, "moe_set_profile_events: event %d is NULL", i);
    L->prof[i] = static_cast<cudaEvent_t>(events[i]);
  }
  L->prof_on = 1;
  return MOE_OK;
}

extern "C" const char* moe_last_error(void) { return g_err; }

// Internal helpers for entry points defined in other translation units.
namespace moe {
int check_scratch(void* ws, cudaStream_t st, const char* name) { return check_workspace(ws, st, name); }
int report_error(int code, const char* msg) { return fail(code, "%s", msg); }
int report_cuda(cudaError_t e, const char* what) { return cuda_fail(e, what); }
int layer_device(const moe_layer* L) { return valid(L) ? L->device : -1; }
const moe_layer_desc* layer_desc(const moe_layer* L) { return valid(L) ? &L->d : nullptr; }
uint64_t layer_record_stride(const moe_layer* L) { return L->off_r.stride; }
uint64_t layer_record_bytes(const moe_layer* L) { return L->off_r.bytes; }

// A decode call's arguments for the expert cache: validated like moe_decode,
// with the routed records read through the cache's slot pool.
int prepare_cached_decode(moe_layer* L, const uint16_t* x, int32_t B, uint16_t* ob, float* of,
                          int32_t* ids, float* wts, void* ws, size_t ws_bytes, const uint8_t* pool,
                          const int32_t* slot_of, const int32_t* slot_tag, int n_slots, LayerArgs* a,
                          bool* single, int* num_sms, const char* name) {
  int rc = prepare(L, x, B, ob, of, ids, wts, ws, ws_bytes, Path::kDecode, false, a, name);
  if (rc || B == 0) return rc;
  a->records = pool, a->slot_of = slot_of, a->slot_tag = slot_tag, a->n_slots = n_slots;
  a->prof_on = 0;
  // residual-VQ layers run their own kernels (never the single-token split)
  *single = L->d.wbits == 4 && B == 1 && plan_b1(*a, L->num_sms, L->smem_optin);
  *num_sms = L->num_sms;
  return MOE_OK;
}

// The router alone (ids and weights), for a routing predicted ahead of the
// layer's own step; no output buffer is needed.
int prepare_route(moe_layer* L, const uint16_t* x, int32_t B, int32_t* ids, float* wts, void* ws,
                  size_t ws_bytes, LayerArgs* a, bool* single, int* num_sms, const char* name) {
  int rc = prepare(L, x, B, nullptr, nullptr, ids, wts, ws, ws_bytes, Path::kRoute, false, a, name);
  if (rc || B == 0) return rc;
  a->prof_on = 0;
  *single = L->d.wbits == 4 && B == 1 && plan_b1(*a, L->num_sms, L->smem_optin);
  *num_sms = L->num_sms;
  return MOE_OK;
}
}  // namespace moe
