// vh_api.cu -- host side of the C interface declared in include/vh.h.
//
// Every entry point validates host scalars and pointer alignment, derives the
// launch plan from the shape and the current device, and launches on the
// caller's stream.  Nothing here synchronises, allocates or reads device
// memory, so the calls can be captured into a CUDA graph (after the first
// call on a device, which sets kernel attributes).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/vh.h"
#include "vh_kernels.h"
#include "vh_plan.h"

namespace {

using vh::AttnParams;
using vh::DeviceInfo;
using vh::WsLayout;
using vh::device_info;
using vh::aligned16;
using vh::valid_shape;
using vh::valid_paging;
using vh::valid_table;
using vh::plan_attn;
using vh::ws_layout;
using vh::encode_cache_maps;
using vh::too_many_tiles;
using vh::kMaxDevices;

// Launch plan, tensor maps and CTA count of an attention launch (p holds the
// shape, element type, cache pointers and strides).  False if the plan or
// the tensor-map encoder rejects the shape.
bool prepare_attn(AttnParams& p, const DeviceInfo& dev, bool fused, int num_ctas) {
  int auto_n = 0;
  if (!plan_attn(p, dev, fused, &auto_n)) return false;
  if (!encode_cache_maps(p)) return false;
  p.N = num_ctas > 0 ? num_ctas : auto_n;
  // the first segment's q rows are requested by thread 0 as soon as the
  // dependency wait returns (measured 0.4-0.5 us faster per launch)
  p.early_q = 1;
  return true;
}

// Point p at the per-step plan region of the workspace (VH_FLAG_PLANNED).
void attach_plan(AttnParams& p, unsigned char* ws, const WsLayout& w, bool planned) {
  p.planned = planned ? 1 : 0;
  p.plan_hdr = reinterpret_cast<const int*>(ws + w.hdr);
  p.plan_rows = reinterpret_cast<const int*>(ws + w.rows);
  p.plan_recs = reinterpret_cast<const int*>(ws + w.recs);
  p.rows_bytes = vh::plan_rows_bytes(p.B);
}

}  // namespace

extern "C" {

const char* vh_status_string(int status) {
  switch (status) {
    case VH_OK: return "ok";
    case VH_EINVAL: return "invalid argument (NULL pointer, unsupported shape or out-of-range scalar)";
    case VH_EALIGN: return "pointer or stride not 16-byte aligned";
    case VH_EWORKSPACE: return "workspace missing or too small";
    case VH_ECUDA: return "CUDA launch error";
    case VH_ENODEV: return "no usable sm_103 device is current";
    case VH_ESCRATCH: return "shape needs more scratch than the built-in fixed scratch array holds";
    default: return "unknown status";
  }
}

int vh_selftest_wait_timeout(int32_t* err_flag, void* stream) {
  if (!err_flag) return VH_EINVAL;
  if ((reinterpret_cast<uintptr_t>(err_flag) & 3u) != 0) return VH_EALIGN;
  if (!device_info()) return VH_ENODEV;
  return vh::launch_wait_timeout_selftest(err_flag, static_cast<cudaStream_t>(stream)) == cudaSuccess ? VH_OK
                                                                                                    : VH_ECUDA;
}

int vh_rope_table(float* cos_sin, int max_pos, int head_dim, double theta, void* stream) {
  if (!cos_sin || max_pos < 1 || (head_dim != 64 && head_dim != 128) || !(theta > 0.0)) return VH_EINVAL;
  if (!aligned16(cos_sin)) return VH_EALIGN;
  if (!device_info()) return VH_ENODEV;
  return vh::launch_rope_table(cos_sin, max_pos, head_dim, theta, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? VH_OK
             : VH_ECUDA;
}

int vh_rope_kv_append(const vh_e16* q, const vh_e16* k_new, const vh_e16* v_new,
                      const float* cos_sin, int max_pos, const int32_t* positions,
                      const float* q_norm_w, const float* k_norm_w, float norm_eps,
                      vh_e16* k_cache, vh_e16* v_cache, int64_t page_stride,
                      int64_t token_stride, int64_t head_stride, int num_pages,
                      const int32_t* page_table, int max_pages_per_seq,
                      const int32_t* seq_lens, const int32_t* active,
                      float* q_rot, int32_t* err_flag, unsigned flags,
                      int B, int Hq, int Hkv, int D, int page_size, void* stream) {
  if (!q || !k_new || !v_new || !cos_sin || !k_cache || !v_cache || !seq_lens || !active || !q_rot ||
      (flags & ~(VH_FLAG_FP16 | VH_FLAG_ROPE_INTERLEAVED)) != 0 || !valid_paging(page_size, max_pages_per_seq) ||
      !valid_table(page_table, B, max_pages_per_seq, num_pages))
    return VH_EINVAL;
  if (!valid_shape(B, Hq, Hkv, D, page_size) || max_pos < 1 || num_pages < 1 || max_pages_per_seq < 1 ||
      page_stride < 1 || token_stride < 1 || head_stride < 1 || too_many_tiles(B, max_pages_per_seq, page_size))
    return VH_EINVAL;
  if (!(norm_eps >= 0.f) || !(norm_eps < 1e30f)) return VH_EINVAL;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(cos_sin) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(q_rot) || (page_stride * 2) % 16 != 0 || (token_stride * 2) % 16 != 0 ||
      (head_stride * 2) % 16 != 0 || !aligned16(q_norm_w) || !aligned16(k_norm_w))
    return VH_EALIGN;
  if (!device_info()) return VH_ENODEV;
  vh::RopeAppendParams p{};
  p.q_norm_w = q_norm_w;
  p.k_norm_w = k_norm_w;
  p.norm_eps = norm_eps;
  p.rope_interleaved = (flags & VH_FLAG_ROPE_INTERLEAVED) != 0;
  p.f16 = (flags & VH_FLAG_FP16) != 0;
  p.q = q;
  p.k_new = k_new;
  p.v_new = v_new;
  p.cos_sin = cos_sin;
  p.max_pos = max_pos;
  p.positions = positions;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.page_stride = page_stride;
  p.token_stride = token_stride;
  p.head_stride = head_stride;
  p.num_pages = num_pages;
  p.page_table = page_table;
  p.max_pages_per_seq = max_pages_per_seq;
  p.seq_lens = seq_lens;
  p.active = active;
  p.q_rot = q_rot;
  p.err_flag = err_flag;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.P = page_size;
  return vh::launch_rope_kv_append(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? VH_OK : VH_ECUDA;
}

int vh_decode_num_ctas(int B, int Hq, int Hkv, int D, int page_size) {
  if (!valid_shape(B, Hq, Hkv, D, page_size)) return VH_EINVAL;
  const DeviceInfo* dev = device_info();
  if (!dev) return VH_ENODEV;
  AttnParams p{};
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.P = page_size;
  int n = 0;
  if (!plan_attn(p, *dev, false, &n)) return VH_EINVAL;
  return n;
}

size_t vh_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int page_size, int num_ctas) {
  if (!valid_shape(B, Hq, Hkv, D, page_size) || num_ctas < 0) return 0;
  int N = num_ctas;
  if (N == 0) {
    // large enough for the automatic CTA count of both the three-call and the
    // fused path, with either element type
    const DeviceInfo* dev = device_info();
    if (!dev) return 0;
    for (bool fused : {false, true})
      for (int f16 : {0, 1}) {
        AttnParams p{};
        p.B = B;
        p.Hq = Hq;
        p.Hkv = Hkv;
        p.D = D;
        p.P = page_size;
        p.f16 = f16;
        int n = 0;
        if (!plan_attn(p, *dev, fused, &n)) return 0;
        N = std::max(N, n);
      }
  }
  return ws_layout(B, Hq, Hkv, D, N).total;
}

int vh_paged_decode_attn(const float* q_rot, const vh_e16* k_cache, const vh_e16* v_cache,
                         int64_t page_stride, int64_t token_stride, int64_t head_stride, int num_pages,
                         const int32_t* page_table, int max_pages_per_seq,
                         const int32_t* seq_lens, const int32_t* active,
                         vh_e16* out, float sm_scale, int num_ctas,
                         void* workspace, size_t workspace_bytes, int32_t* err_flag, unsigned flags,
                         int B, int Hq, int Hkv, int D, int page_size, void* stream) {
  if (!q_rot || !k_cache || !v_cache || !seq_lens || !active || !out ||
      (flags & ~(VH_FLAG_FP16 | VH_FLAG_PDL | VH_FLAG_PLANNED)) != 0 || !valid_paging(page_size, max_pages_per_seq) ||
      !valid_table(page_table, B, max_pages_per_seq, num_pages))
    return VH_EINVAL;
  if (!valid_shape(B, Hq, Hkv, D, page_size) || num_pages < 1 || max_pages_per_seq < 1 || page_stride < 1 ||
      token_stride < 1 || head_stride < 1 || num_ctas < 0 || num_ctas > 65535 ||
      too_many_tiles(B, max_pages_per_seq, page_size) || !(sm_scale == sm_scale))
    return VH_EINVAL;
  if (!aligned16(q_rot) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (page_stride * 2) % 16 != 0 || (token_stride * 2) % 16 != 0 || (head_stride * 2) % 16 != 0)
    return VH_EALIGN;
  if (!workspace) return VH_EWORKSPACE;
  if (!aligned16(workspace)) return VH_EALIGN;
  const DeviceInfo* dev = device_info();
  if (!dev) return VH_ENODEV;
  AttnParams p{};
  p.q_rot = q_rot;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.page_stride = page_stride;
  p.token_stride = token_stride;
  p.head_stride = head_stride;
  p.num_pages = num_pages;
  p.page_table = page_table;
  p.max_pages_per_seq = max_pages_per_seq;
  p.seq_lens = seq_lens;
  p.active = active;
  p.out = out;
  p.err_flag = err_flag;
  p.f16 = (flags & VH_FLAG_FP16) != 0;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.P = page_size;
  if (!prepare_attn(p, *dev, false, num_ctas)) return VH_EINVAL;
  const WsLayout w = ws_layout(B, Hq, Hkv, D, p.N);
  if (workspace_bytes < w.total) return VH_EWORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  p.plan = reinterpret_cast<int4*>(ws + w.plan);
  p.part_lse = reinterpret_cast<float*>(ws + w.lse);
  p.part_o = reinterpret_cast<float*>(ws + w.o);
  attach_plan(p, ws, w, (flags & VH_FLAG_PLANNED) != 0);
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf(static_cast<float>(D));
  p.scale_log2 = scale * 1.4426950408889634f;
  return vh::launch_decode_attn(p, static_cast<cudaStream_t>(stream), (flags & VH_FLAG_PDL) != 0) == cudaSuccess
             ? VH_OK
             : VH_ECUDA;
}

int vh_decode_combine(const void* workspace, size_t workspace_bytes, vh_e16* out, int num_ctas,
                      unsigned flags, int B, int Hq, int Hkv, int D, int page_size, void* stream) {
  if (!out || !valid_shape(B, Hq, Hkv, D, page_size) || num_ctas < 0 || num_ctas > 65535 ||
      (flags & ~static_cast<unsigned>(VH_FLAG_FP16)) != 0)
    return VH_EINVAL;
  if (!aligned16(out)) return VH_EALIGN;
  if (!workspace) return VH_EWORKSPACE;
  if (!aligned16(workspace)) return VH_EALIGN;
  const DeviceInfo* dev = device_info();
  if (!dev) return VH_ENODEV;
  AttnParams a{};
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.P = page_size;
  a.f16 = (flags & VH_FLAG_FP16) != 0;  // the attention launch's plan: same element type
  int auto_n = 0;
  if (!plan_attn(a, *dev, false, &auto_n)) return VH_EINVAL;
  const int N = num_ctas > 0 ? num_ctas : auto_n;
  const WsLayout w = ws_layout(B, Hq, Hkv, D, N);
  if (workspace_bytes < w.total) return VH_EWORKSPACE;
  const unsigned char* ws = static_cast<const unsigned char*>(workspace);
  vh::CombineParams p{};
  p.plan = reinterpret_cast<const int4*>(ws + w.plan);
  p.part_lse = reinterpret_cast<const float*>(ws + w.lse);
  p.part_o = reinterpret_cast<const float*>(ws + w.o);
  p.out = out;
  p.B = B;
  p.Hq = Hq;
  p.D = D;
  p.Hc = a.Hc;
  p.G = a.G;
  p.N = N;
  p.f16 = (flags & VH_FLAG_FP16) != 0;
  return vh::launch_decode_combine(p, a.groups, static_cast<cudaStream_t>(stream)) == cudaSuccess ? VH_OK
                                                                                                 : VH_ECUDA;
}

int vh_decode_fused(const vh_e16* q, const vh_e16* k_new, const vh_e16* v_new,
                    const float* cos_sin, int max_pos, const int32_t* positions,
                    const float* q_norm_w, const float* k_norm_w, float norm_eps,
                    vh_e16* k_cache, vh_e16* v_cache, int64_t page_stride, int64_t token_stride,
                    int64_t head_stride, int num_pages, const int32_t* page_table, int max_pages_per_seq,
                    const int32_t* seq_lens, const int32_t* active,
                    vh_e16* out, float sm_scale, int num_ctas,
                    void* workspace, size_t workspace_bytes, int32_t* err_flag, unsigned flags,
                    int B, int Hq, int Hkv, int D, int page_size, void* stream) {
  if (!q || !k_new || !v_new || !cos_sin || !k_cache || !v_cache || !seq_lens || !active || !out ||
      (flags & ~(VH_FLAG_PDL | VH_FLAG_PDL_KV | VH_FLAG_FP16 | VH_FLAG_ROPE_INTERLEAVED | VH_FLAG_PLANNED |
                 VH_FLAG_HOST_IO)) != 0 ||
      !valid_paging(page_size, max_pages_per_seq) || !valid_table(page_table, B, max_pages_per_seq, num_pages))
    return VH_EINVAL;
  if (!valid_shape(B, Hq, Hkv, D, page_size) || max_pos < 1 || num_pages < 1 || max_pages_per_seq < 1 ||
      page_stride < 1 || token_stride < 1 || head_stride < 1 || num_ctas < 0 || num_ctas > 65535 ||
      too_many_tiles(B, max_pages_per_seq, page_size) || !(sm_scale == sm_scale))
    return VH_EINVAL;
  if (!(norm_eps >= 0.f) || !(norm_eps < 1e30f)) return VH_EINVAL;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(cos_sin) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(out) || (page_stride * 2) % 16 != 0 || (token_stride * 2) % 16 != 0 ||
      (head_stride * 2) % 16 != 0 || !aligned16(q_norm_w) || !aligned16(k_norm_w))
    return VH_EALIGN;
  if (!workspace) return VH_EWORKSPACE;
  if (!aligned16(workspace)) return VH_EALIGN;
  const DeviceInfo* dev = device_info();
  if (!dev) return VH_ENODEV;
  AttnParams p{};
  p.q_norm_w = q_norm_w;
  p.k_norm_w = k_norm_w;
  p.norm_eps = norm_eps;
  p.rope_interleaved = (flags & VH_FLAG_ROPE_INTERLEAVED) != 0;
  p.f16 = (flags & VH_FLAG_FP16) != 0;
  p.q = q;
  p.k_new = k_new;
  p.v_new = v_new;
  p.cos_sin = cos_sin;
  p.max_pos = max_pos;
  p.positions = positions;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_cache_w = k_cache;
  p.v_cache_w = v_cache;
  p.page_stride = page_stride;
  p.token_stride = token_stride;
  p.head_stride = head_stride;
  p.num_pages = num_pages;
  p.page_table = page_table;
  p.max_pages_per_seq = max_pages_per_seq;
  p.seq_lens = seq_lens;
  p.active = active;
  p.out = out;
  p.err_flag = err_flag;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.P = page_size;
  if (!prepare_attn(p, *dev, true, num_ctas)) return VH_EINVAL;
  const WsLayout w = ws_layout(B, Hq, Hkv, D, p.N);
  if (workspace_bytes < w.total) return VH_EWORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  p.plan = reinterpret_cast<int4*>(ws + w.plan);
  p.counters = reinterpret_cast<int*>(ws + w.counters);
  p.part_lse = reinterpret_cast<float*>(ws + w.lse);
  p.part_o = reinterpret_cast<float*>(ws + w.o);
  attach_plan(p, ws, w, (flags & VH_FLAG_PLANNED) != 0);
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf(static_cast<float>(D));
  p.scale_log2 = scale * 1.4426950408889634f;
  p.prefetch_kv = (flags & VH_FLAG_PDL_KV) != 0;
  if (flags & VH_FLAG_HOST_IO) {
    p.host_io = 1;
    p.q_tx_bytes = D * 4;  // only the RoPE row arrives by bulk copy
  }
  // with the first stages requested before the wait (launches without it measured slower)
  p.l2_tiles = p.prefetch_kv ? vh::l2_prefetch_tiles() : 0;
  return vh::launch_decode_attn(p, static_cast<cudaStream_t>(stream),
                                (flags & (VH_FLAG_PDL | VH_FLAG_PDL_KV)) != 0) == cudaSuccess
             ? VH_OK
             : VH_ECUDA;
}

int vh_decode_plan(const int32_t* positions, int max_pos, int num_pages, const int32_t* page_table,
                   int max_pages_per_seq, const int32_t* seq_lens, const int32_t* active, int num_ctas,
                   void* workspace, size_t workspace_bytes, int32_t* err_flag, unsigned flags,
                   int B, int Hq, int Hkv, int D, int page_size, void* stream) {
  if (!seq_lens || !active || (flags & ~(VH_FLAG_FP16 | VH_FLAG_PLAN_THREE_CALL)) != 0 ||
      !valid_paging(page_size, max_pages_per_seq) || !valid_table(page_table, B, max_pages_per_seq, num_pages))
    return VH_EINVAL;
  const bool fused = (flags & VH_FLAG_PLAN_THREE_CALL) == 0;
  if (!valid_shape(B, Hq, Hkv, D, page_size) || num_pages < 1 || max_pages_per_seq < 1 || num_ctas < 0 ||
      num_ctas > 65535 || too_many_tiles(B, max_pages_per_seq, page_size) || (fused && max_pos < 1))
    return VH_EINVAL;
  if (!workspace) return VH_EWORKSPACE;
  if (!aligned16(workspace)) return VH_EALIGN;
  const DeviceInfo* dev = device_info();
  if (!dev) return VH_ENODEV;
  AttnParams a{};
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.P = page_size;
  a.f16 = (flags & VH_FLAG_FP16) != 0;
  int auto_n = 0;
  if (!plan_attn(a, *dev, fused, &auto_n)) return VH_EINVAL;
  const int N = num_ctas > 0 ? num_ctas : auto_n;
  const WsLayout w = ws_layout(B, Hq, Hkv, D, N);
  if (workspace_bytes < w.total) return VH_EWORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  vh::PlanParams p{};
  p.seq_lens = seq_lens;
  p.active = active;
  p.positions = positions;
  p.page_table = page_table;
  p.max_pages_per_seq = max_pages_per_seq;
  p.max_pos = max_pos;
  p.P = page_size;
  p.B = B;
  p.N = N;
  p.min_tiles = a.min_tiles;
  p.fused = fused ? 1 : 0;
  p.hdr = reinterpret_cast<int*>(ws + w.hdr);
  p.rows = reinterpret_cast<int*>(ws + w.rows);
  p.recs = reinterpret_cast<int*>(ws + w.recs);
  vh::plan_rows_bytes(B, &p.len_idx, &p.pos_idx);
  p.err_flag = err_flag;
  return vh::launch_decode_plan(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? VH_OK : VH_ECUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Attention without caller-provided scratch.
//
// Some callers have no way to allocate device memory for the workspace: code
// running under an allocator they do not control (a serving runtime that
// hands kernels only preallocated arenas), plug-ins whose host process owns
// the CUDA context, or tools that must not change the memory footprint
// between two measurements.  For them the split-K partial results go into
// one fixed array that lives in this library's device image.  Every GPU
// that loads the library keeps it, VH_STATIC_SCRATCH_BYTES bytes, until the
// process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_static_scratch[VH_STATIC_SCRATCH_BYTES];

namespace {

// Device address of g_static_scratch on each device, once a lookup succeeded.
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of the fixed scratch array on the current device, looked up
// with that device current.  In host code the array's name is only a
// host-side stand-in and must never be handed to a kernel.  Only a successful
// lookup is kept: after a failed one (for instance a first call made during
// a stream capture) the next call tries again.
void* static_scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_static_ptr[dev] = p;
  }
  return g_static_ptr[dev];
}

}  // namespace

extern "C" int vh_paged_decode_attn_noalloc(const float* q_rot, const vh_bf16* k_cache, const vh_bf16* v_cache,
                                            int64_t page_stride, int64_t token_stride, int num_pages,
                                            const int32_t* page_table, int max_pages_per_seq,
                                            const int32_t* seq_lens, const int32_t* active,
                                            vh_bf16* out, float sm_scale, int num_ctas, int32_t* err_flag,
                                            int B, int Hq, int Hkv, int D, int page_size, void* stream) {
  if (!q_rot || !k_cache || !v_cache || !seq_lens || !active || !out ||
      !valid_paging(page_size, max_pages_per_seq) || !valid_table(page_table, B, max_pages_per_seq, num_pages))
    return VH_EINVAL;
  if (!valid_shape(B, Hq, Hkv, D, page_size) || num_pages < 1 || max_pages_per_seq < 1 || page_stride < 1 ||
      token_stride < 1 || num_ctas < 0 || num_ctas > 65535 || too_many_tiles(B, max_pages_per_seq, page_size) ||
      !(sm_scale == sm_scale))
    return VH_EINVAL;
  if (!aligned16(q_rot) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (page_stride * 2) % 16 != 0 || (token_stride * 2) % 16 != 0)
    return VH_EALIGN;
  const DeviceInfo* dev = device_info();
  if (!dev) return VH_ENODEV;
  AttnParams p{};
  p.q_rot = q_rot;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.page_stride = page_stride;
  p.token_stride = token_stride;
  p.head_stride = D;  // token-major pages: the heads of a slot are contiguous
  p.num_pages = num_pages;
  p.page_table = page_table;
  p.max_pages_per_seq = max_pages_per_seq;
  p.seq_lens = seq_lens;
  p.active = active;
  p.out = out;
  p.err_flag = err_flag;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.P = page_size;
  if (!prepare_attn(p, *dev, false, num_ctas)) return VH_EINVAL;
  const WsLayout w = ws_layout(B, Hq, Hkv, D, p.N);
  if (w.total > static_cast<size_t>(VH_STATIC_SCRATCH_BYTES)) return VH_ESCRATCH;
  unsigned char* ws = static_cast<unsigned char*>(static_scratch_address());
  if (!ws) return VH_ECUDA;
  // Nothing in the scratch has to start at zero: the attention kernel writes
  // the per-row plan and every partial result before the combine reads them.
  p.plan = reinterpret_cast<int4*>(ws + w.plan);
  p.part_lse = reinterpret_cast<float*>(ws + w.lse);
  p.part_o = reinterpret_cast<float*>(ws + w.o);
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf(static_cast<float>(D));
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (vh::launch_decode_attn(p, st, false) != cudaSuccess) return VH_ECUDA;
  vh::CombineParams c{};
  c.plan = p.plan;
  c.part_lse = p.part_lse;
  c.part_o = p.part_o;
  c.out = out;
  c.B = B;
  c.Hq = Hq;
  c.D = D;
  c.Hc = p.Hc;
  c.G = p.G;
  c.N = p.N;
  return vh::launch_decode_combine(c, p.groups, st) == cudaSuccess ? VH_OK : VH_ECUDA;
}
