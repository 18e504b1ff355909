// moe_api.cu — the C ABI (include/moe_nvfp4.h): argument validation, the expert pack, the
// workspace layout and the launch sequence of the NVFP4 routed-expert MoE step on sm_103a.
#include "../../include/moe_nvfp4.h"
#include "moe_internal.cuh"

#include <cmath>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

namespace moe {
size_t route_narrow_smem_bytes(int T, int H, int E, int k);
void* noalloc_scratch_of_current_device();
}

struct moe_expert_pack {
  int E, H, I, device;
  unsigned char* buf;
  size_t bytes;
  moe::PackView view;
  float x_scale;
  float x_inv6S;
  int x_scale_uniform;
  std::vector<float> mult_h;      // [E][3]
  std::vector<float> in_scale_h;  // [E][3]
};

namespace {

thread_local int g_last_launches = 0;
// One-shot per-launch profiling of the next forward call on this thread (see LaunchProf), and
// the kernels the last profiled call launched.
thread_local moe::LaunchProf g_prof = {};
thread_local const void* g_prof_funcs[32] = {nullptr};
thread_local int g_prof_nfuncs = 0;

// Ends a profiled call: keeps its kernel list and switches profiling off.
void prof_finish() {
  if (g_prof.count == 0) return;
  g_prof_nfuncs = g_prof.next < 32 ? g_prof.next : 32;
  for (int i = 0; i < g_prof_nfuncs; ++i) g_prof_funcs[i] = g_prof.func[i];
  g_prof.count = 0;
  g_prof.next = 0;
}

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool finite_pos(float v) { return std::isfinite(v) && v > 0.0f; }

// fl32(1 / fl32(6 * S)), evaluated with IEEE single-precision operations.
float inv6S_of(float S) {
  volatile float six_s = 6.0f * S;
  volatile float r = 1.0f / six_s;
  return r;
}

int num_sms_of_current_device() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

struct WsLayout {
  size_t ctl, gmeta, slot_amax, logits, idx, w, slot_of, counts, offsets, perm,
      chunk_base, xh, xfac, xq, xsf, h16, hq, hsf, y, htag, ytag, xres, tt_expert, tt_slot0, tt_n, ttbase, xq_perm,
      xsf_atoms, hq_perm, hsf_atoms, xh_perm, hf_perm, sh_hs, sh_sigma, sh_y, sh_gu, sh_tag, total;
  size_t sh_tag_bytes;
  size_t slot_amax_bytes;
  int G, NT;
};

// mode: 0 W4A16, 1 W4A4, 2 W4A8, -1 routing only (no expert buffers). Is > 0 adds the shared
// expert's buffers after everything else, so the other offsets do not depend on it.
WsLayout ws_layout(int T, int H, int E, int k, int I, int mode, int Is = 0) {
  WsLayout L;
  const long long S = (long long)T * k;
  L.G = (int)((S + moe::kGroup - 1) / moe::kGroup + (S < E ? S : E));
  const int nchunk = (T + 31) / 32;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
  L.ctl = take(moe::kCtlWords * 4);
  L.gmeta = take((size_t)L.G * sizeof(moe::GroupMeta));
  L.slot_amax_bytes = mode == 0 ? (size_t)S * 4 : 0;
  L.slot_amax = take(L.slot_amax_bytes);
  const bool narrow = T <= moe::kNarrowT;
  L.logits = take((size_t)T * E * (narrow ? 8 * moe::kLogitReplicas : 4));
  L.idx = take((size_t)S * 4);
  L.w = take((size_t)S * 4);
  L.slot_of = take((size_t)S * 4);
  L.counts = take((size_t)E * 4);
  L.offsets = take((size_t)(E + 1) * 4);
  L.perm = take((size_t)S * 4);
  L.chunk_base = take(T > moe::kNarrowT ? (size_t)nchunk * E * 4 : 0);
  L.xh = take(mode >= 0 ? (size_t)T * H * 2 : 0);
  L.xfac = take(mode >= 0 ? (size_t)T * 4 : 0);
  L.xq = take(mode == 1 ? (size_t)T * H / 2 : mode == 2 ? (size_t)T * H : 0);
  L.xsf = take(mode == 1 ? (size_t)T * H / 16 : 0);
  L.h16 = take(mode == 0 ? (size_t)S * I * 2 : 0);
  L.hq = take(mode == 1 ? (size_t)S * I / 2 : mode == 2 ? (size_t)S * I : 0);
  L.hsf = take(mode == 1 ? (size_t)S * I / 16 : 0);
  L.y = take(mode >= 0 ? (size_t)S * H * 2 : 0);
  L.htag = take(mode >= 0 && narrow ? (size_t)S * (I / 16) * 9 * 8 : 0);
  L.ytag = take(mode >= 0 && narrow ? (size_t)S * (H / 2) * 8 : 0);
  // grouped tensor-core path (wide calls): 128-slot token tiles in a padded permuted space
  const bool tc = mode >= 0 && moe::tile_path(T, H, I, mode);
  L.NT = tc ? (int)((S + 127) / 128 + (S < E ? S : E)) : 0;
  const size_t P = (size_t)L.NT * 128;
  const bool w4a4 = tc && mode == 1, w4a16 = tc && (mode == 0 || mode == 2);
  L.tt_expert = take((size_t)L.NT * 4);
  L.tt_slot0 = take((size_t)L.NT * 4);
  L.tt_n = take((size_t)L.NT * 4);
  L.ttbase = take(tc ? (size_t)(E + 1) * 4 : 0);
  L.xq_perm = take(w4a4 ? P * H / 2 : 0);
  L.xsf_atoms = take(w4a4 ? (size_t)L.NT * (H / 64) * 512 : 0);
  L.hq_perm = take(w4a4 ? P * I / 2 : 0);
  L.hsf_atoms = take(w4a4 ? (size_t)L.NT * (I / 64 > 0 ? I / 64 : 1) * 512 : 0);
  L.xh_perm = take(w4a16 ? P * H * 2 : 0);
  L.hf_perm = take(w4a16 ? P * I * 2 : 0);
  L.sh_hs = take(Is > 0 ? (size_t)T * Is * 2 : 0);
  L.sh_sigma = take(Is > 0 ? (size_t)T * 4 : 0);
  L.sh_y = take(Is > 0 ? (size_t)T * H * 4 : 0);
  L.sh_gu = take(Is > 0 && !narrow ? (size_t)T * 2 * Is * 4 : 0);
  L.sh_tag_bytes = Is > 0 && narrow ? ((size_t)T * Is + T + (size_t)T * H) * 8 : 0;
  L.sh_tag = take(L.sh_tag_bytes);
  // a layer of a chained stack: the next layer's input (this layer's input + output)
  L.xres = take(mode >= 0 ? (size_t)T * H * 2 : 0);
  L.total = o;
  return L;
}

moe::WsView ws_view(void* ws, const WsLayout& L, int T, int H, int E, int k, int I) {
  unsigned char* b = static_cast<unsigned char*>(ws);
  moe::WsView v;
  v.ctl = reinterpret_cast<uint32_t*>(b + L.ctl);
  v.gmeta = reinterpret_cast<moe::GroupMeta*>(b + L.gmeta);
  v.slot_amax = L.slot_amax_bytes ? reinterpret_cast<uint32_t*>(b + L.slot_amax) : nullptr;
  v.logits = reinterpret_cast<float*>(b + L.logits);
  v.idx = reinterpret_cast<int32_t*>(b + L.idx);
  v.w = reinterpret_cast<float*>(b + L.w);
  v.slot_of = reinterpret_cast<int32_t*>(b + L.slot_of);
  v.counts = reinterpret_cast<int32_t*>(b + L.counts);
  v.offsets = reinterpret_cast<int32_t*>(b + L.offsets);
  v.perm = reinterpret_cast<int32_t*>(b + L.perm);
  v.chunk_base = reinterpret_cast<int32_t*>(b + L.chunk_base);
  v.xh = reinterpret_cast<__half*>(b + L.xh);
  v.xfac = reinterpret_cast<float*>(b + L.xfac);
  v.xq = b + L.xq;
  v.xsf = b + L.xsf;
  v.h16 = reinterpret_cast<uint16_t*>(b + L.h16);
  v.hq = b + L.hq;
  v.hsf = b + L.hsf;
  v.y = reinterpret_cast<uint16_t*>(b + L.y);
  v.htag = reinterpret_cast<unsigned long long*>(b + L.htag);
  v.ytag = reinterpret_cast<unsigned long long*>(b + L.ytag);
  v.T = T; v.H = H; v.E = E; v.k = k; v.I = I; v.G = L.G; v.NT = L.NT;
  const bool tc = L.NT > 0;
  v.tt_expert = tc ? reinterpret_cast<int32_t*>(b + L.tt_expert) : nullptr;
  v.tt_slot0 = reinterpret_cast<int32_t*>(b + L.tt_slot0);
  v.tt_n = reinterpret_cast<int32_t*>(b + L.tt_n);
  v.ttbase = reinterpret_cast<int32_t*>(b + L.ttbase);
  v.xq_perm = b + L.xq_perm;
  v.xsf_atoms = b + L.xsf_atoms;
  v.hq_perm = b + L.hq_perm;
  v.hsf_atoms = b + L.hsf_atoms;
  v.xh_perm = reinterpret_cast<__half*>(b + L.xh_perm);
  v.hf_perm = reinterpret_cast<__half*>(b + L.hf_perm);
  v.sh_y = nullptr;
  v.sh_sigma = nullptr;
  v.sh_tag = L.sh_tag_bytes ? reinterpret_cast<unsigned long long*>(b + L.sh_tag) : nullptr;
  return v;
}

// Device allocation of moe_pack_nvfp4; fails on request of the test fault injection.
cudaError_t pack_alloc(void** p, size_t bytes) {
  moe::FaultInjection& fi = moe::fault_injection();
  if (fi.fail_pack_allocs > 0) {
    --fi.fail_pack_allocs;
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMalloc(p, bytes);
}

moe_status from_cuda(cudaError_t e) {
  return e == cudaSuccess ? MOE_OK : (e == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA);
}

bool mode_ok(int mode) { return mode == MOE_W4A16 || mode == MOE_W4A4 || mode == MOE_W4A8; }

// W4A8 runs on the fused narrow kernel and on the wide tcgen05 f16 path only
bool a8_supported(int T, int H, int E, int k, int I) {
  if (T <= moe::kNarrowT)
    return moe::decode_geom(T, H, E, k, I, num_sms_of_current_device(), nullptr);
  return moe::tile_path(T, H, I, 2);
}

bool route_shape_ok(int T, int H, int E, int k) {
  return T >= 1 && T <= 65536 && H >= 128 && H % 128 == 0 && H <= 8192 && E >= 1 && E <= 1024 &&
         k >= 1 && k <= E && k <= 32;
}

// Layout of the last call on each workspace (by address). The fused narrow kernel's epoch-tagged
// words (logits, h, Y) rely on their regions holding zeros or tagged words of earlier calls; a
// call of another layout (shape, mode, pack dimensions, shared expert, layer count) puts other
// data at those offsets, whose upper halves can equal a later call's epoch. So the first fused
// call after a layout change clears its tagged regions (a memset on the call's stream).
uint64_t layout_sig(int kind, int T, int H, int E, int k, int I, int mode, int Is, int layers) {
  uint64_t h = 1469598103934665603ull;   // FNV-1a over the fields
  for (long long f : {(long long)kind, (long long)T, (long long)H, (long long)E, (long long)k,
                      (long long)I, (long long)mode, (long long)Is, (long long)layers}) {
    h ^= (uint64_t)f;
    h *= 1099511628211ull;
  }
  return h;
}

// Records sig as the workspace's layout; true when the workspace held another layout before.
bool layout_changed(const void* ws, uint64_t sig) {
  static std::mutex mu;
  static std::unordered_map<const void*, uint64_t> last;
  std::lock_guard<std::mutex> g(mu);
  auto it = last.find(ws);
  if (it == last.end()) {
    last.emplace(ws, sig);
    return false;   // a workspace is zero-filled before its first use
  }
  const bool changed = it->second != sig;
  it->second = sig;
  return changed;
}

// Clears the tagged regions of a narrow call's layout at byte offset base of the workspace.
cudaError_t clear_tags(unsigned char* ws, size_t base, const WsLayout& L, int T, int H, int E,
                       int k, int I, cudaStream_t s) {
  const size_t S = (size_t)T * k;
  const size_t parts[4][2] = {{L.logits, (size_t)T * E * 8 * moe::kLogitReplicas},
                              {L.htag, S * (I / 16) * 9 * 8},
                              {L.ytag, S * (H / 2) * 8},
                              {L.sh_tag, L.sh_tag_bytes}};
  for (const auto& p : parts) {
    const cudaError_t e = cudaMemsetAsync(ws + base + p[0], 0, p[1], s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Chained layers: the control words, then one region per layer laid out as a single call's
// workspace without its control words.
size_t layer_stride(const WsLayout& L) { return L.total - L.gmeta; }
size_t layers_total(const WsLayout& L, int layers) { return L.gmeta + layers * layer_stride(L); }

// The view of layer l's region (control words shared), as the kernels' own layer view.
moe::WsView shift_view(moe::WsView v, size_t off) {
  auto mv = [&](auto*& p) { moe::shift_ptr(p, off); };
  mv(v.gmeta); mv(v.slot_amax); mv(v.logits); mv(v.idx); mv(v.w); mv(v.slot_of); mv(v.counts);
  mv(v.offsets); mv(v.perm); mv(v.chunk_base); mv(v.xh); mv(v.xfac); mv(v.xq); mv(v.xsf);
  mv(v.h16); mv(v.hq); mv(v.hsf); mv(v.y); mv(v.htag); mv(v.ytag); mv(v.tt_expert);
  mv(v.tt_slot0); mv(v.tt_n); mv(v.ttbase); mv(v.xq_perm); mv(v.xsf_atoms); mv(v.hq_perm);
  mv(v.hsf_atoms); mv(v.xh_perm); mv(v.hf_perm);
  return v;
}

}  // namespace

namespace moe {
LaunchProf& launch_prof() { return g_prof; }
FaultInjection& fault_injection() {
  static FaultInjection fi = {0, -1, 0};
  return fi;
}
}  // namespace moe

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_OOM: return "MOE_ERR_OOM";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
  }
  return "MOE_ERR_UNKNOWN";
}

int moe_last_launch_count(void) { return g_last_launches; }

moe_status moe_profile_next_forward(void* const* events, int count) {
  if (count < 0 || count > 64 || (count > 0 && !events)) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) g_prof.ev[i] = static_cast<cudaEvent_t>(events[i]);
  g_prof.count = count;
  g_prof.next = 0;
  return MOE_OK;
}

moe_status moe_test_inject_faults(int skip_logits_cta, double wait_limit_seconds,
                                  int fail_pack_allocations) {
  if (skip_logits_cta < -1 || !(wait_limit_seconds >= 0.0) || wait_limit_seconds > 10.0 ||
      fail_pack_allocations < 0)
    return MOE_ERR_INVALID_ARG;
  moe::FaultInjection& fi = moe::fault_injection();
  fi.skip_logits_cta = skip_logits_cta;
  fi.wait_ns = (uint64_t)(wait_limit_seconds * 1e9);
  fi.fail_pack_allocs = fail_pack_allocations;
  return MOE_OK;
}

const char* moe_profile_kernel_name(int i) {
  if (i < 0 || i >= g_prof_nfuncs || !g_prof_funcs[i]) return nullptr;
  const char* name = nullptr;
  if (cudaFuncGetName(&name, g_prof_funcs[i]) != cudaSuccess) return nullptr;
  return name;
}

moe_status moe_pack_nvfp4(const moe_nvfp4_matrix* gate, const moe_nvfp4_matrix* up,
                          const moe_nvfp4_matrix* down, int num_experts, int hidden, int inter,
                          void* stream, moe_expert_pack** out) {
  if (!gate || !up || !down || !out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  const int E = num_experts, H = hidden, I = inter;
  if (E < 1 || E > 1024 || H < 128 || H % 128 || H > 8192 || I < 64 || I % 64 || I > 2048)
    return MOE_ERR_INVALID_ARG;
  for (int e = 0; e < E; ++e) {
    const moe_nvfp4_matrix* m[3] = {&gate[e], &up[e], &down[e]};
    for (auto* p : m)
      if (!p->codes || !p->scales || !finite_pos(p->multiplier) || !finite_pos(p->input_scale))
        return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t mat_codes = (size_t)I * H / 2;   // codes of one gate/up/down matrix
  const size_t mat_scales = (size_t)I * H / 16;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
  const size_t off_gc = take(mat_codes * E), off_uc = take(mat_codes * E),
               off_dc = take(mat_codes * E), off_gus = take(2 * mat_scales * E),
               off_ds = take(mat_scales * E), off_agu = take(2 * mat_scales * E),
               off_adn = take(mat_scales * E), off_mult = take((size_t)E * 12),
               off_dsc = take((size_t)E * 4), off_dinv = take((size_t)E * 4);
  moe_expert_pack* pk = new (std::nothrow) moe_expert_pack();
  if (!pk) return MOE_ERR_OOM;
  pk->E = E; pk->H = H; pk->I = I;
  cudaGetDevice(&pk->device);
  pk->bytes = o;
  if (pack_alloc(reinterpret_cast<void**>(&pk->buf), o) != cudaSuccess) {
    cudaGetLastError();
    delete pk;
    return MOE_ERR_OOM;
  }
  unsigned char* raw = nullptr;
  if (pack_alloc(reinterpret_cast<void**>(&raw), 3 * mat_scales * E) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(pk->buf);
    delete pk;
    return MOE_ERR_OOM;
  }
  cudaError_t err = cudaSuccess;
  for (int e = 0; e < E && err == cudaSuccess; ++e) {
    err = cudaMemcpyAsync(pk->buf + off_gc + e * mat_codes, gate[e].codes, mat_codes,
                          cudaMemcpyDefault, s);
    if (err == cudaSuccess)
      err = cudaMemcpyAsync(pk->buf + off_uc + e * mat_codes, up[e].codes, mat_codes,
                            cudaMemcpyDefault, s);
    if (err == cudaSuccess)
      err = cudaMemcpyAsync(pk->buf + off_dc + e * mat_codes, down[e].codes, mat_codes,
                            cudaMemcpyDefault, s);
    if (err == cudaSuccess)
      err = cudaMemcpyAsync(raw + e * mat_scales, gate[e].scales, mat_scales, cudaMemcpyDefault, s);
    if (err == cudaSuccess)
      err = cudaMemcpyAsync(raw + (E + e) * mat_scales, up[e].scales, mat_scales,
                            cudaMemcpyDefault, s);
    if (err == cudaSuccess)
      err = cudaMemcpyAsync(raw + (2 * E + e) * mat_scales, down[e].scales, mat_scales,
                            cudaMemcpyDefault, s);
  }
  pk->mult_h.resize((size_t)E * 3);
  pk->in_scale_h.resize((size_t)E * 3);
  std::vector<float> dsc(E), dinv(E);
  pk->x_scale = gate[0].input_scale;
  pk->x_scale_uniform = 1;
  for (int e = 0; e < E; ++e) {
    pk->mult_h[e * 3 + 0] = gate[e].multiplier;
    pk->mult_h[e * 3 + 1] = up[e].multiplier;
    pk->mult_h[e * 3 + 2] = down[e].multiplier;
    pk->in_scale_h[e * 3 + 0] = gate[e].input_scale;
    pk->in_scale_h[e * 3 + 1] = up[e].input_scale;
    pk->in_scale_h[e * 3 + 2] = down[e].input_scale;
    if (gate[e].input_scale != pk->x_scale || up[e].input_scale != pk->x_scale)
      pk->x_scale_uniform = 0;
    dsc[e] = down[e].input_scale;
    dinv[e] = inv6S_of(down[e].input_scale);
  }
  pk->x_inv6S = inv6S_of(pk->x_scale);
  if (err == cudaSuccess)
    err = moe::launch_pack_scales(s, raw, raw + E * mat_scales, raw + 2 * E * mat_scales, E, H, I,
                                  pk->buf + off_gus, pk->buf + off_ds, pk->buf + off_agu,
                                  pk->buf + off_adn);
  if (err == cudaSuccess)
    err = cudaMemcpyAsync(pk->buf + off_mult, pk->mult_h.data(), (size_t)E * 12,
                          cudaMemcpyHostToDevice, s);
  if (err == cudaSuccess)
    err = cudaMemcpyAsync(pk->buf + off_dsc, dsc.data(), (size_t)E * 4, cudaMemcpyHostToDevice, s);
  if (err == cudaSuccess)
    err = cudaMemcpyAsync(pk->buf + off_dinv, dinv.data(), (size_t)E * 4, cudaMemcpyHostToDevice, s);
  cudaError_t se = cudaStreamSynchronize(s);
  if (err == cudaSuccess) err = se;
  cudaFree(raw);
  if (err != cudaSuccess) {
    cudaFree(pk->buf);
    delete pk;
    return from_cuda(err);
  }
  moe::PackView& v = pk->view;
  v.gate_codes = pk->buf + off_gc;
  v.up_codes = pk->buf + off_uc;
  v.down_codes = pk->buf + off_dc;
  v.gu_scales = pk->buf + off_gus;
  v.down_scales = pk->buf + off_ds;
  v.mult = reinterpret_cast<const float*>(pk->buf + off_mult);
  v.down_in_scale = reinterpret_cast<const float*>(pk->buf + off_dsc);
  v.down_inv6S = reinterpret_cast<const float*>(pk->buf + off_dinv);
  v.sfa_gu = pk->buf + off_agu;
  v.sfa_down = pk->buf + off_adn;
  v.E = E; v.H = H; v.I = I;
  *out = pk;
  return MOE_OK;
}

moe_status moe_pack_destroy(moe_expert_pack* pack) {
  if (!pack) return MOE_OK;
  cudaError_t e = cudaFree(pack->buf);
  delete pack;
  return from_cuda(e);
}

moe_status moe_pack_info(const moe_expert_pack* pack, int* num_experts, int* hidden, int* inter,
                         size_t* device_bytes) {
  if (!pack) return MOE_ERR_INVALID_ARG;
  if (num_experts) *num_experts = pack->E;
  if (hidden) *hidden = pack->H;
  if (inter) *inter = pack->I;
  if (device_bytes) *device_bytes = pack->bytes;
  return MOE_OK;
}

moe_status moe_pack_get_matrix(const moe_expert_pack* pack, int expert, int which, uint8_t* codes,
                               uint8_t* scales, float* multiplier, float* input_scale) {
  if (!pack || expert < 0 || expert >= pack->E || which < 0 || which > 2 || !codes || !scales)
    return MOE_ERR_INVALID_ARG;
  const size_t mat_codes = (size_t)pack->I * pack->H / 2;
  const size_t mat_scales = (size_t)pack->I * pack->H / 16;
  const uint8_t* src = which == 0 ? pack->view.gate_codes
                       : which == 1 ? pack->view.up_codes : pack->view.down_codes;
  cudaError_t e = cudaMemcpy(codes, src + expert * mat_codes, mat_codes, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return from_cuda(e);
  unsigned char* tmp = nullptr;
  if (cudaMalloc(&tmp, mat_scales) != cudaSuccess) { cudaGetLastError(); return MOE_ERR_OOM; }
  e = moe::launch_unpack_scales(0, pack->view.gu_scales, pack->view.down_scales, pack->E, pack->H,
                                pack->I, expert, which, tmp);
  if (e == cudaSuccess) e = cudaMemcpy(scales, tmp, mat_scales, cudaMemcpyDeviceToHost);
  cudaFree(tmp);
  if (multiplier) *multiplier = pack->mult_h[expert * 3 + which];
  if (input_scale) *input_scale = pack->in_scale_h[expert * 3 + which];
  return from_cuda(e);
}

moe_status moe_workspace_size(const moe_expert_pack* pack, int T, int k, moe_mode mode,
                              size_t* bytes) {
  if (!pack || !bytes || !mode_ok(mode) ||
      !route_shape_ok(T, pack->H, pack->E, k))
    return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(T, pack->H, pack->E, k, pack->I, (int)mode).total;
  return MOE_OK;
}

moe_status moe_route_workspace_size(int T, int H, int E, int k, size_t* bytes) {
  if (!bytes || !route_shape_ok(T, H, E, k)) return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(T, H, E, k, 0, -1).total;
  return MOE_OK;
}

moe_status moe_workspace_offsets(const moe_expert_pack* pack, int T, int k, moe_mode mode,
                                 moe_ws_offsets* off) {
  if (!pack || !off || !mode_ok(mode) ||
      !route_shape_ok(T, pack->H, pack->E, k))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(T, pack->H, pack->E, k, pack->I, (int)mode);
  off->idx = L.idx; off->w = L.w; off->counts = L.counts; off->offsets = L.offsets;
  off->perm = L.perm; off->slot_of = L.slot_of; off->x_codes = L.xq; off->x_scales = L.xsf;
  off->h_bf16 = L.h16; off->h_codes = L.hq; off->h_scales = L.hsf; off->y = L.y;
  return MOE_OK;
}

moe_status moe_route_topk(const uint16_t* x, const uint16_t* router_w, int T, int H, int E, int k,
                          int32_t* idx, float* w, int32_t* counts, int32_t* offsets, int32_t* perm,
                          void* ws, size_t ws_bytes, void* stream) {
  g_last_launches = 0;
  if (!x || !router_w || !idx || !w || !counts || !offsets || !perm || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (!route_shape_ok(T, H, E, k)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(T, H, E, k, 0, -1);
  (void)layout_changed(ws, layout_sig(0, T, H, E, k, 0, -1, 0, 1));
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  moe::WsView v = ws_view(ws, L, T, H, E, k, 0);
  moe::LaunchCfg lc{static_cast<cudaStream_t>(stream), num_sms_of_current_device(), true};
  cudaError_t e;
  if (T <= moe::kNarrowT) {
    e = moe::launch_route_narrow(lc, x, router_w, v, nullptr, -1, 1.0f, 1.0f, idx, w, counts,
                                 offsets, perm);
    g_last_launches = 1;
  } else {
    int n = 0;
    e = moe::launch_route_wide(lc, x, router_w, v, nullptr, idx, w, counts, offsets, perm, &n);
    g_last_launches = n;
  }
  return from_cuda(e);
}

}  // extern "C"

namespace {

bool shared_ok(const moe_shared_expert* sh, int H) {
  return sh && sh->gate_up && sh->down && sh->gate && aligned16(sh->gate_up) &&
         aligned16(sh->down) && aligned16(sh->gate) && sh->inter >= 64 && sh->inter % 64 == 0 &&
         sh->inter <= 2048 && H % 64 == 0;
}

// The launch sequence of one call on a prepared workspace view: the shared expert first (when
// given; its buffers at the offsets of L in the workspace at `wsb`), then the routed step on the
// fused narrow kernel, the multi-kernel narrow path or the grouped wide path. Adds the kernels
// launched to *n.
cudaError_t launch_forward(moe::LaunchCfg lc, const moe_expert_pack* pack,
                           const moe_shared_expert* sh, const WsLayout& L, unsigned char* wsb,
                           moe::WsView v, int m, const uint16_t* x, const uint16_t* router_w,
                           uint16_t* out, int* n) {
  const int T = v.T, H = v.H, E = v.E, k = v.k, I = v.I;
  const bool narrow = T <= moe::kNarrowT;
  cudaError_t e = cudaSuccess;
  moe::ShView sv{};
  if (sh) {
    sv.gate_up = sh->gate_up;
    sv.down = sh->down;
    sv.gate = sh->gate;
    sv.hs = reinterpret_cast<uint16_t*>(wsb + L.sh_hs);
    sv.sigma = reinterpret_cast<float*>(wsb + L.sh_sigma);
    sv.ys = reinterpret_cast<float*>(wsb + L.sh_y);
    sv.gu = reinterpret_cast<float*>(wsb + L.sh_gu);
    sv.Is = sh->inter;
  }
  const bool fused_ok = narrow && moe::decode_geom(T, H, E, k, I, lc.num_sms, nullptr);
  if (sh && fused_ok && T <= 2 && v.sh_tag) {
    // one or two tokens: the shared expert inside the fused kernel (its weight rows stream while
    // the router's logits are exchanged), unless the shape leaves it no room
    const cudaError_t d = moe::launch_decode(lc, pack->view, v, m, pack->x_scale, pack->x_inv6S,
                                             x, router_w, out, nullptr, &sv);
    if (d != cudaErrorNotSupported && d != cudaErrorCooperativeLaunchTooLarge) {
      *n += 1;
      return d;
    }
    cudaGetLastError();
  }
  if (sh) {
    // the shared expert first: the combine (of whichever path runs) adds its term
    e = moe::launch_shared(lc, x, sv, v, n);
    v.sh_y = sv.ys;
    v.sh_sigma = sv.sigma;
  }
  if (fused_ok) {
    // the whole routed step in one persistent kernel (unless its CTAs cannot all be resident)
    if (e == cudaSuccess) {
      const cudaError_t d = moe::launch_decode(lc, pack->view, v, m, pack->x_scale,
                                               pack->x_inv6S, x, router_w, out, nullptr);
      if (d != cudaErrorCooperativeLaunchTooLarge) {
        *n += 1;
        return d;
      }
      cudaGetLastError();
    } else {
      return e;
    }
  }
  if (narrow) {
    if (e == cudaSuccess)
      e = moe::launch_route_narrow(lc, x, router_w, v, &pack->view, m, pack->x_scale,
                                   pack->x_inv6S, v.idx, v.w, v.counts, v.offsets, v.perm);
    *n += 1;
  }
  // wide calls run the tensor-core grouped path when the layout reserved its token tiles
  const bool use_tc = !narrow && v.NT > 0;
  if (!narrow) {
    if (e == cudaSuccess)
      e = moe::launch_route_wide(lc, x, router_w, v, &pack->view, v.idx, v.w, v.counts, v.offsets,
                                 v.perm, n);
    if (e == cudaSuccess && !use_tc) {   // the tensor-core path quantises x itself
      e = moe::launch_xprep_wide(lc, x, v, m, pack->x_scale, pack->x_inv6S);
      *n += 1;
    }
  }
  if (use_tc) {
    // x operand by padded slot, gate/up, (h operand,) down on tcgen05
    if (e == cudaSuccess) {
      if (m == 1) {
        e = moe::launch_tc_experts(lc, pack->view, v, x, pack->x_scale, pack->x_inv6S);
        *n += 3;
      } else {
        e = moe::launch_tc16_experts(lc, pack->view, v, x, m == 2, pack->x_scale, pack->x_inv6S);
        *n += 4;
      }
    }
  } else {
    if (e == cudaSuccess) {
      e = moe::launch_gateup(lc, pack->view, v, m, narrow);
      *n += 1;
    }
    if (e == cudaSuccess) {
      const long long S = (long long)T * k;
      const bool h_res = narrow && S * (2LL * I + 16) <= 96 * 1024;
      e = moe::launch_down(lc, pack->view, v, m, h_res);
      *n += 1;
    }
  }
  if (e == cudaSuccess) {
    e = moe::launch_combine(lc, v, out);
    *n += 1;
  }
  return e;
}

// moe_forward, optionally with the shared expert (validated by the caller).
moe_status forward_impl(const uint16_t* x, const uint16_t* router_w, const moe_expert_pack* pack,
                        const moe_shared_expert* sh, int T, int k, moe_mode mode, uint16_t* out,
                        void* ws, size_t ws_bytes, void* stream) {
  g_last_launches = 0;
  if (!x || !router_w || !pack || !out || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(out) || !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  if (!mode_ok(mode)) return MOE_ERR_INVALID_ARG;
  const int H = pack->H, E = pack->E, I = pack->I;
  if (!route_shape_ok(T, H, E, k)) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<const void*>(out) == reinterpret_cast<const void*>(x))
    return MOE_ERR_INVALID_ARG;
  if (mode != MOE_W4A16 && !pack->x_scale_uniform) return MOE_ERR_UNSUPPORTED;
  if (mode == MOE_W4A8 && !a8_supported(T, H, E, k, I)) return MOE_ERR_UNSUPPORTED;
  const bool narrow = T <= moe::kNarrowT;
  if (sh && !narrow && !moe::tc_supported()) return MOE_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(T, H, E, k, I, (int)mode, sh ? sh->inter : 0);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  moe::WsView v = ws_view(ws, L, T, H, E, k, I);
  moe::LaunchCfg lc{static_cast<cudaStream_t>(stream), num_sms_of_current_device(), true};
  // while profiling, launches are not overlapped by programmatic dependent launch
  if (g_prof.count) lc.pdl = false;
  if (layout_changed(ws, layout_sig(sh ? 2 : 1, T, H, E, k, I, (int)mode, sh ? sh->inter : 0, 1)) &&
      narrow) {
    const cudaError_t ce = clear_tags(static_cast<unsigned char*>(ws), 0, L, T, H, E, k, I, lc.stream);
    if (ce != cudaSuccess) return from_cuda(ce);
  }
  int n = 0;
  const cudaError_t e = launch_forward(lc, pack, sh, L, static_cast<unsigned char*>(ws), v,
                                       (int)mode, x, router_w, out, &n);
  prof_finish();
  g_last_launches = n;
  return from_cuda(e);
}

}  // namespace

extern "C" {

moe_status moe_forward(const uint16_t* x, const uint16_t* router_w, const moe_expert_pack* pack,
                       int T, int k, moe_mode mode, uint16_t* out, void* ws, size_t ws_bytes,
                       void* stream) {
  return forward_impl(x, router_w, pack, nullptr, T, k, mode, out, ws, ws_bytes, stream);
}

moe_status moe_workspace_size_layers(const moe_expert_pack* pack, int layers, int T, int k,
                                     moe_mode mode, size_t* bytes) {
  if (!pack || !bytes || layers < 1 || !mode_ok(mode) ||
      !route_shape_ok(T, pack->H, pack->E, k))
    return MOE_ERR_INVALID_ARG;
  *bytes = layers_total(ws_layout(T, pack->H, pack->E, k, pack->I, (int)mode), layers);
  return MOE_OK;
}

moe_status moe_workspace_offsets_layers(const moe_expert_pack* pack, int layers, int T, int k,
                                        moe_mode mode, int layer, moe_ws_offsets* off) {
  if (layer < 0 || layer >= layers) return MOE_ERR_INVALID_ARG;
  const moe_status st = moe_workspace_offsets(pack, T, k, mode, off);
  if (st != MOE_OK) return st;
  const size_t d = (size_t)layer *
                   layer_stride(ws_layout(T, pack->H, pack->E, k, pack->I, (int)mode));
  off->idx += d; off->w += d; off->counts += d; off->offsets += d; off->perm += d;
  off->slot_of += d; off->x_codes += d; off->x_scales += d; off->h_bf16 += d; off->h_codes += d;
  off->h_scales += d; off->y += d;
  return MOE_OK;
}

moe_status moe_forward_layers(const uint16_t* x, const uint16_t* const* router_w,
                              const moe_expert_pack* const* packs, int layers, int T, int k,
                              moe_mode mode, uint16_t* out, void* ws, size_t ws_bytes,
                              void* stream) {
  g_last_launches = 0;
  if (!x || !router_w || !packs || !out || !ws || layers < 1) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (!mode_ok(mode)) return MOE_ERR_INVALID_ARG;
  const moe_expert_pack* p0 = packs[0];
  if (!p0) return MOE_ERR_INVALID_ARG;
  const int H = p0->H, E = p0->E, I = p0->I;
  if (!route_shape_ok(T, H, E, k)) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < layers; ++l) {
    if (!packs[l] || !router_w[l] || !aligned16(router_w[l])) return MOE_ERR_INVALID_ARG;
    if (packs[l]->H != H || packs[l]->E != E || packs[l]->I != I) return MOE_ERR_INVALID_ARG;
    if (mode != MOE_W4A16 && !packs[l]->x_scale_uniform) return MOE_ERR_UNSUPPORTED;
  }
  if (mode == MOE_W4A8 && !a8_supported(T, H, E, k, I)) return MOE_ERR_UNSUPPORTED;
  const size_t act = (size_t)T * H;   // elements of one layer's activations
  const uint16_t* xe = x + act;
  if (xe > out && x < out + layers * act) return MOE_ERR_INVALID_ARG;   // x overlaps out
  const WsLayout L = ws_layout(T, H, E, k, I, (int)mode);
  if (ws_bytes < layers_total(L, layers)) return MOE_ERR_WORKSPACE;
  const size_t stride = layer_stride(L);
  const moe::WsView v0 = ws_view(ws, L, T, H, E, k, I);
  moe::LaunchCfg lc{static_cast<cudaStream_t>(stream), num_sms_of_current_device(), true};
  if (g_prof.count) lc.pdl = false;
  if (layout_changed(ws, layout_sig(3, T, H, E, k, I, (int)mode, 0, layers)) &&
      T <= moe::kNarrowT) {
    for (int l = 0; l < layers; ++l) {
      const cudaError_t ce = clear_tags(static_cast<unsigned char*>(ws), (size_t)l * stride, L,
                                        T, H, E, k, I, lc.stream);
      if (ce != cudaSuccess) return from_cuda(ce);
    }
  }
  const int m = (int)mode;
  cudaError_t e = cudaSuccess;
  int n = 0;
  unsigned char* wsb = static_cast<unsigned char*>(ws);
  // the residual sum x + out of layer l, in its region: the input of layer l + 1
  auto xres_of = [&](int l) {
    return reinterpret_cast<uint16_t*>(wsb + L.xres + (size_t)l * stride);
  };
  if (T <= moe::kNarrowT && moe::decode_geom(T, H, E, k, I, lc.num_sms, nullptr)) {
    // one launch of the fused kernel per layer, chained by programmatic dependent launch: each
    // launch copies its router rows before waiting for the previous one, and its combine also
    // writes the residual sum, the next launch's input
    for (int l = 0; l < layers && e == cudaSuccess; ++l) {
      const moe_expert_pack* p = packs[l];
      e = moe::launch_decode(lc, p->view, shift_view(v0, (size_t)l * stride), m, p->x_scale,
                             p->x_inv6S, l == 0 ? x : xres_of(l - 1), router_w[l],
                             out + (size_t)l * act, l + 1 < layers ? xres_of(l) : nullptr);
      n += 1;
    }
  } else {
    // the same chain as one launch sequence per layer, each in its own workspace region, and
    // the residual sum between them
    for (int l = 0; l < layers && e == cudaSuccess; ++l) {
      const uint16_t* xl = l == 0 ? x : xres_of(l - 1);
      e = launch_forward(lc, packs[l], nullptr, L, wsb, shift_view(v0, (size_t)l * stride), m,
                         xl, router_w[l], out + (size_t)l * act, &n);
      if (e == cudaSuccess && l + 1 < layers) {
        e = moe::launch_residual_add(lc, xl, out + (size_t)l * act, xres_of(l), act);
        n += 1;
      }
    }
  }
  prof_finish();
  g_last_launches = n;
  return from_cuda(e);
}

moe_status moe_workspace_size_shared(const moe_expert_pack* pack, int T, int k, moe_mode mode,
                                     int shared_inter, size_t* bytes) {
  if (!pack || !bytes || !mode_ok(mode) ||
      !route_shape_ok(T, pack->H, pack->E, k) || shared_inter < 64 || shared_inter % 64 ||
      shared_inter > 2048)
    return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(T, pack->H, pack->E, k, pack->I, (int)mode, shared_inter).total;
  return MOE_OK;
}

moe_status moe_workspace_offsets_shared(const moe_expert_pack* pack, int T, int k, moe_mode mode,
                                        int shared_inter, size_t* h, size_t* sigma, size_t* y) {
  size_t bytes = 0;
  const moe_status st = moe_workspace_size_shared(pack, T, k, mode, shared_inter, &bytes);
  if (st != MOE_OK) return st;
  const WsLayout L = ws_layout(T, pack->H, pack->E, k, pack->I, (int)mode, shared_inter);
  if (h) *h = L.sh_hs;
  if (sigma) *sigma = L.sh_sigma;
  if (y) *y = L.sh_y;
  return MOE_OK;
}

moe_status moe_forward_shared(const uint16_t* x, const uint16_t* router_w,
                              const moe_expert_pack* pack, const moe_shared_expert* shared, int T,
                              int k, moe_mode mode, uint16_t* out, void* ws, size_t ws_bytes,
                              void* stream) {
  g_last_launches = 0;
  if (!pack || !shared_ok(shared, pack->H)) return MOE_ERR_INVALID_ARG;
  return forward_impl(x, router_w, pack, shared, T, k, mode, out, ws, ws_bytes, stream);
}

moe_status moe_quantize_act_nvfp4(const uint16_t* x, int rows, int cols, float input_scale,
                                  uint8_t* codes, uint8_t* scales, void* stream) {
  if (!x || !codes || !scales || rows < 1 || cols < 16 || cols % 16 || !finite_pos(input_scale))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(codes) & 7u)) return MOE_ERR_INVALID_ARG;
  moe::LaunchCfg lc{static_cast<cudaStream_t>(stream), num_sms_of_current_device(), true};
  return from_cuda(moe::launch_quantize_rows(lc, x, rows, cols, input_scale, inv6S_of(input_scale),
                                             codes, scales));
}

moe_status moe_read_device_status(void* ws, void* stream, moe_status* status) {
  if (!status) return MOE_ERR_INVALID_ARG;
  if (!ws) {   // the fixed array of moe_route_topk_noalloc on the current device
    ws = moe::noalloc_scratch_of_current_device();
    if (!ws) return MOE_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  uint32_t* word = static_cast<uint32_t*>(ws) + moe::kCtlStatus;
  cudaError_t e = cudaMemcpyAsync(&v, word, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(word, 0, 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return from_cuda(e);
  *status = static_cast<moe_status>(v);
  return MOE_OK;
}

}  // extern "C"
