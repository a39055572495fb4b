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
using vh::auto_ctas;
using vh::ws_layout;
using vh::encode_cache_maps;
using vh::too_many_tiles;
using vh::kMaxDevices;

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
  if (!plan_attn(p, *dev, false)) return VH_EINVAL;
  return auto_ctas(p, *dev);
}

size_t vh_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int page_size, int num_ctas) {
  if (!valid_shape(B, Hq, Hkv, D, page_size) || num_ctas < 0) return 0;
  int N = num_ctas;
  if (N == 0) {
    // large enough for the automatic CTA count of both the three-call and the fused path
    const DeviceInfo* dev = device_info();
    if (!dev) return 0;
    for (bool fused : {false, true}) {
      AttnParams p{};
      p.B = B;
      p.Hq = Hq;
      p.Hkv = Hkv;
      p.D = D;
      p.P = page_size;
      if (!plan_attn(p, *dev, fused)) return 0;
      N = std::max(N, auto_ctas(p, *dev));
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
      (flags & ~(VH_FLAG_FP16 | VH_FLAG_PDL)) != 0 || !valid_paging(page_size, max_pages_per_seq) ||
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
  if (!plan_attn(p, *dev, false)) return VH_EINVAL;
  if (!encode_cache_maps(p)) return VH_EINVAL;
  p.N = num_ctas > 0 ? num_ctas : auto_ctas(p, *dev);
  const WsLayout w = ws_layout(B, Hq, Hkv, D, p.N);
  if (workspace_bytes < w.total) return VH_EWORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  p.plan = reinterpret_cast<int4*>(ws + w.plan);
  p.part_lse = reinterpret_cast<float*>(ws + w.lse);
  p.part_o = reinterpret_cast<float*>(ws + w.o);
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf(static_cast<float>(D));
  p.scale_log2 = scale * 1.4426950408889634f;
  p.early_q = vh::env_int("VH_DECODE_EARLY_Q", 1) != 0;
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
  if (!plan_attn(a, *dev, false)) return VH_EINVAL;
  const int N = num_ctas > 0 ? num_ctas : auto_ctas(a, *dev);
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
      (flags & ~(VH_FLAG_PDL | VH_FLAG_PDL_KV | VH_FLAG_FP16 | VH_FLAG_ROPE_INTERLEAVED)) != 0 ||
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
  if (!plan_attn(p, *dev, true)) return VH_EINVAL;
  if (!encode_cache_maps(p)) return VH_EINVAL;
  p.N = num_ctas > 0 ? num_ctas : auto_ctas(p, *dev);
  const WsLayout w = ws_layout(B, Hq, Hkv, D, p.N);
  if (workspace_bytes < w.total) return VH_EWORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  p.plan = reinterpret_cast<int4*>(ws + w.plan);
  p.counters = reinterpret_cast<int*>(ws + w.counters);
  p.part_lse = reinterpret_cast<float*>(ws + w.lse);
  p.part_o = reinterpret_cast<float*>(ws + w.o);
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf(static_cast<float>(D));
  p.scale_log2 = scale * 1.4426950408889634f;
  p.early_q = vh::env_int("VH_DECODE_EARLY_Q", 1) != 0;
  p.prefetch_kv = (flags & VH_FLAG_PDL_KV) != 0;
  // with the first stages requested before the wait (launches without it measured slower)
  p.l2_tiles = p.prefetch_kv ? vh::l2_prefetch_tiles() : 0;
  return vh::launch_decode_attn(p, static_cast<cudaStream_t>(stream),
                                (flags & (VH_FLAG_PDL | VH_FLAG_PDL_KV)) != 0) == cudaSuccess
             ? VH_OK
             : VH_ECUDA;
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

struct StaticScratch {
  std::once_flag once;
  void* ptr = nullptr;  // device address of g_static_scratch on this device
};
StaticScratch g_static[kMaxDevices];

// Device address of the fixed scratch array on the current device.  Resolved
// once per device, with that device current; in host code the array's name is
// only a host-side stand-in and must never be handed to a kernel.
void* static_scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  StaticScratch& s = g_static[dev];
  std::call_once(s.once, [&]() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    s.ptr = p;
  });
  return s.ptr;
}

}  // namespace

extern "C" int vh_paged_decode_attn_noalloc(const float* q_rot, const vh_bf16* k_cache, const vh_bf16* v_cache,
                                            int64_t page_stride, int64_t token_stride, int num_pages,
                                            const int32_t* page_table, int max_pages_per_seq,
                                            const int32_t* seq_lens, const int32_t* active,
                                            vh_bf16* out, float sm_scale, int num_ctas, int32_t* err_flag,
                                            int B, int Hq, int Hkv, int D, int page_size, void* stream) {
  if (!q_rot || !k_cache || !v_cache || !page_table || !seq_lens || !active || !out ||
      !valid_paging(page_size, max_pages_per_seq))
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
  if (!plan_attn(p, *dev, false)) return VH_EINVAL;
  if (!encode_cache_maps(p)) return VH_EINVAL;
  p.N = num_ctas > 0 ? num_ctas : auto_ctas(p, *dev);
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
