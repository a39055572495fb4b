// vh_api.cu -- host side of the C interface declared in include/vh.h.
//
// Every entry point validates host scalars and pointer alignment, derives the
// launch plan from the shape and the current device, and launches on the
// caller's stream.  Nothing here synchronises, allocates or reads device
// memory, so the calls can be captured into a CUDA graph (after the first
// call on a device, which sets kernel attributes).
#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include "../../include/vh.h"
#include "vh_kernels.h"

namespace {

using vh::AttnParams;

constexpr int kMaxDevices = 64;
constexpr int kMaxStages = 8;
// Lower bound on tiles per CTA when the work list is short.  One tile: a
// short list (the Fast AR step: 64 one-tile rows) then spreads over as many
// CTAs as it has tiles, which measured 2.1x faster there than four tiles per
// CTA and the same on the long lists (VH_DECODE_MIN_TILES, for tuning).
constexpr int kMinTilesPerCta = 1;

struct DeviceInfo {
  std::once_flag once;
  bool ok = false;
  int sm_count = 0;
  int smem_optin = 0;
};
DeviceInfo g_dev[kMaxDevices];

const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  DeviceInfo& d = g_dev[dev];
  std::call_once(d.once, [&]() {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    // The kernels are built for sm_103a only.
    if (major != 10 || minor != 3) return;
    for (int D : {64, 128})
      for (int G : {1, 2, 4, 8})
        if (vh::prepare_decode_attn(D, G, d.smem_optin) != cudaSuccess) {
          cudaGetLastError();
          return;
        }
    d.ok = true;
  });
  return d.ok ? &d : nullptr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_gqa(int Hq, int Hkv) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return false;
  const int G = Hq / Hkv;
  return G == 1 || G == 2 || G == 4 || G == 8;
}

bool valid_shape(int B, int Hq, int Hkv, int D, int P) {
  return B >= 1 && B <= 65535 && valid_gqa(Hq, Hkv) && (D == 64 || D == 128) && P >= 1 && P <= 1024 &&
         Hkv <= 1024;
}

// Pages of a row hold whole 16-token tiles, unless a row has a single page.
bool valid_paging(int P, int max_pages_per_seq) {
  return max_pages_per_seq >= 1 && (P % 16 == 0 || max_pages_per_seq == 1);
}

// Without a page table, row b's pages are b * max_pages_per_seq + j: they must exist.
bool valid_table(const int32_t* page_table, int B, int max_pages_per_seq, int num_pages) {
  return page_table != nullptr || static_cast<long long>(B) * max_pages_per_seq <= num_pages;
}

int env_int(const char* name, int dflt) {
  const char* s = std::getenv(name);
  if (!s || !*s) return dflt;
  return std::atoi(s);
}

// kv heads per CTA: the largest divisor of Hkv with Hc * D <= 512 (4 heads at
// head_dim 128, 8 at 64): 32 KB tiles, so that two CTAs share an SM and the
// work list is cut twice as fine as with whole-SM CTAs (VH_DECODE_HC sets
// another cap, up to Hc * D <= 1024 and Hc <= 8, for tuning).
int choose_hc(int Hkv, int D) {
  int cap = std::min(512 / D, 8);
  const int want = env_int("VH_DECODE_HC", 0);
  if (want >= 1) cap = std::min(want, std::min(1024 / D, 8));
  int hc = std::min(Hkv, cap);
  while (Hkv % hc != 0) --hc;
  return hc;
}

// Pipeline stages per CTA.  Two stages of 32 KB per CTA (128 KB in flight
// per SM with two CTAs) keep HBM saturated on GB300; more bytes in flight
// only lengthen the queues, which measured slower at the start and the end
// of a launch (VH_DECODE_STAGES sets another count, for tuning).
constexpr int kDefaultStages = 2;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared-memory plan of the attention kernel (fused or not): kDefaultStages
// pipeline stages (or VH_DECODE_STAGES, if they fit); if two stages do not
// fit, fewer kv heads go to each CTA.  Returns false if even one head per CTA
// cannot have two stages.
bool plan_attn(AttnParams& p, const DeviceInfo& dev, bool fused) {
  p.fused = fused ? 1 : 0;
  p.G = p.Hq / p.Hkv;
  const size_t budget = static_cast<size_t>(dev.smem_optin);
  int hc = choose_hc(p.Hkv, p.D);
  size_t fixed = 0;
  int stages = 0;
  for (;;) {
    p.Hc = hc;
    // K and V of a 16-token tile, as swizzled 16 x 128-byte boxes (no padding
    // needed for conflict-free ldmatrix): 2 * 16 * Hc * D * 2 bytes, a
    // multiple of 2048 so every box stays 1024-byte aligned
    p.stage_bytes = 2 * 16 * hc * p.D * 2;
    const size_t hg = static_cast<size_t>(hc) * p.G;
    // staged q rows, contiguous: one bulk copy per segment
    p.q_row_bytes = fused ? p.D * 2 : p.D * 4;
    p.q_tx_bytes = static_cast<int>(fused ? hg * p.D * 2 + p.D * 4 : hg * p.D * 4);
    p.q_bytes = static_cast<int>(hg * p.q_row_bytes + (fused ? p.D * 4 : 0));
    const size_t qs_bytes = fused ? static_cast<size_t>(hc) * p.G * (p.D * 4 + 32) : 0;
    fixed = align_up(p.q_bytes, 128) + align_up(qs_bytes, 128) + align_up(4 * (static_cast<size_t>(p.B) + 1), 16) +
            2 * align_up(4 * static_cast<size_t>(p.B), 16) + 8 * kMaxStages + 8 * (2 * kMaxStages + 4) + 48 * 4 + 256 +
            1024 /* alignment of the base */;
    stages = fixed < budget ? static_cast<int>(std::min<size_t>(kMaxStages, (budget - fixed) / p.stage_bytes)) : 0;
    if (stages >= 2 || hc == 1) break;
    int next = hc - 1;
    while (next > 1 && p.Hkv % next != 0) --next;
    hc = next;
  }
  if (stages < 2) return false;
  p.groups = p.Hkv / p.Hc;
  const int want = env_int("VH_DECODE_STAGES", kDefaultStages);
  if (want >= 2 && want < stages) stages = want;
  p.stages = stages;
  size_t off = static_cast<size_t>(stages) * p.stage_bytes;
  p.q_off = static_cast<int>(off);
  off += align_up(p.q_bytes, 128);
  p.qs_off = static_cast<int>(off);
  if (fused) off += align_up(static_cast<size_t>(p.Hc) * p.G * (p.D * 4 + 32), 128);
  p.cum_off = static_cast<int>(off);
  off += align_up(4 * (static_cast<size_t>(p.B) + 1), 16);
  p.len_off = static_cast<int>(off);
  off += align_up(4 * static_cast<size_t>(p.B), 16);
  p.pos_off = static_cast<int>(off);
  off += align_up(4 * static_cast<size_t>(p.B), 16);
  p.meta_off = static_cast<int>(off);
  off += 8 * static_cast<size_t>(stages);
  p.bar_off = static_cast<int>(align_up(off, 16));
  off = p.bar_off + 8 * (2 * static_cast<size_t>(stages) + 4) + 48 * 4;
  // + up to 1024 bytes that the kernel skips to align its base for the boxes
  p.smem_bytes = static_cast<int>(align_up(off, 128) + 1024);
  p.min_tiles = std::max(1, env_int("VH_DECODE_MIN_TILES", kMinTilesPerCta));
  return static_cast<size_t>(p.smem_bytes) <= budget;
}

int auto_ctas(const AttnParams& p, const DeviceInfo& dev) {
  int per_sm = 0;
  if (vh::decode_attn_occupancy(p, &per_sm) != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  const int want = env_int("VH_DECODE_CTAS_PER_SM", 0);
  if (want >= 1 && want < per_sm) per_sm = want;
  return std::max(1, dev.sm_count * per_sm / p.groups);
}

// Workspace: per-row split plan (int4 [B]); per-(head group, row) counters of
// the fused merge (int [Hkv][B], an upper bound on groups); partial lse
// [groups][N][2][Hq/groups] and partial outputs [...][D] (groups * Hq/groups == Hq).
struct WsLayout {
  size_t plan, counters, lse, o, total;
};

WsLayout ws_layout(int B, int Hq, int Hkv, int D, int N) {
  WsLayout w;
  w.plan = 0;
  w.counters = align_up(static_cast<size_t>(B) * 16, 256);
  w.lse = w.counters + align_up(static_cast<size_t>(B) * Hkv * 4, 256);
  w.o = w.lse + align_up(static_cast<size_t>(N) * 2 * Hq * 4, 256);
  w.total = w.o + static_cast<size_t>(N) * 2 * Hq * D * 4;
  return w;
}

// The driver's tensor-map encoder, looked up once through the runtime (the
// library does not link the driver library itself).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, []() {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

// Tensor maps of the K and V caches for the attention kernel's tile copies:
// 4-D tensors of 16-bit elements (dimension 0 = head_dim, 3 = page) with the
// 128-byte swizzle, boxes of 64 elements x 8 tokens x box_heads heads, which
// land in shared memory as [head][token][128 bytes].  Preferred: dimension
// 1 = token, 2 = head and box_heads = Hc, so a tile is two boxes (token
// groups) per 64-column block of K and of V.  If the encoder rejects that order (the strides of
// token-major pages decrease from dimension 1 to 2), dimensions 1 and 2 are
// token and head in increasing stride order and each box holds one head.
// Sets p.tm_tok_dim and p.box_heads.  Returns false if no encoding is accepted.
bool encode_cache_maps(AttnParams& p) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  // L2 fill granularity of the tile reads (VH_TMA_L2 = 0, 64, 128 or 256 bytes, for tuning)
  CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  switch (env_int("VH_TMA_L2", 256)) {
    case 0: promo = CU_TENSOR_MAP_L2_PROMOTION_NONE; break;
    case 64: promo = CU_TENSOR_MAP_L2_PROMOTION_L2_64B; break;
    case 128: promo = CU_TENSOR_MAP_L2_PROMOTION_L2_128B; break;
    default: break;
  }
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  auto encode = [&](bool tok_first, cuuint32_t heads) -> bool {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(p.D), static_cast<cuuint64_t>(tok_first ? p.P : p.Hkv),
                                static_cast<cuuint64_t>(tok_first ? p.Hkv : p.P),
                                static_cast<cuuint64_t>(p.num_pages)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(2 * (tok_first ? p.token_stride : p.head_stride)),
                                   static_cast<cuuint64_t>(2 * (tok_first ? p.head_stride : p.token_stride)),
                                   static_cast<cuuint64_t>(2 * p.page_stride)};
    const cuuint32_t box[4] = {64, tok_first ? 8u : 1u, tok_first ? heads : 8u, 1};
    for (int kv = 0; kv < 2; ++kv) {
      CUtensorMap* m = kv ? &p.tmap_v : &p.tmap_k;
      void* base = const_cast<uint16_t*>(kv ? p.v_cache : p.k_cache);
      if (enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    }
    p.tm_tok_dim = tok_first ? 1 : 2;
    p.box_heads = static_cast<int>(heads);
    return true;
  };
  if (env_int("VH_TMA_BOX_HEADS", 0) != 1 && encode(true, static_cast<cuuint32_t>(p.Hc))) return true;
  return encode(p.token_stride <= p.head_stride, 1);
}

bool too_many_tiles(int B, int max_pages_per_seq, int P) {
  const long long max_len = static_cast<long long>(max_pages_per_seq) * P;
  return max_len > (1LL << 24) || static_cast<long long>(B) * ((max_len + 15) / 16) >= (1LL << 31);
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
      (flags & ~static_cast<unsigned>(VH_FLAG_FP16)) != 0 || !valid_paging(page_size, max_pages_per_seq) ||
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
  return vh::launch_decode_attn(p, static_cast<cudaStream_t>(stream), false) == cudaSuccess ? VH_OK : VH_ECUDA;
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
  p.prefetch_kv = (flags & VH_FLAG_PDL_KV) != 0;
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
