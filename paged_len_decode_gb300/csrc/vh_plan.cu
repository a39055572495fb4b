// vh_plan.cu -- launch planning of the decode kernels (host side).
//
// Per device: the checks and kernel attributes set once.  Per call: kv heads
// per CTA, pipeline stages and the shared-memory layout, the CTA count, the
// workspace layout, and the tensor maps of the K and V caches.  The entry
// points in vh_api.cu validate arguments and call these.
#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <unordered_map>

#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include "vh_plan.h"

namespace vh {

namespace {
constexpr int kMaxStages = 8;
// Lower bound on tiles per CTA when the work list is short.  One tile: a
// short list (the Fast AR step: 64 one-tile rows) then spreads over as many
// CTAs as it has tiles, which measured 2.1x faster there than four tiles per
// CTA and the same on the long lists.
constexpr int kMinTilesPerCta = 1;
}  // namespace

DeviceInfo g_dev[kMaxDevices];

const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  DeviceInfo& d = g_dev[dev];
  std::call_once(d.once, [&]() {
    d.index = dev;
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
    if (vh::prepare_decode_plan(d.smem_optin) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    d.ok = true;
  });
  return d.ok ? &d : nullptr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool valid_gqa(int Hq, int Hkv) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return false;
  const int G = Hq / Hkv;
  return G == 1 || G == 2 || G == 4 || G == 8;
}

bool valid_shape(int B, int Hq, int Hkv, int D, int P) {
  return B >= 1 && B <= 65535 && valid_gqa(Hq, Hkv) && (D == 64 || D == 128) && P >= 1 && P <= 1024 &&
         Hkv <= 1024;
}

// Pages of a row hold whole 16-token tiles, or exactly half of one (P = 8:
// every tile then spans two pages), unless a row has a single page.
bool valid_paging(int P, int max_pages_per_seq) {
  return max_pages_per_seq >= 1 && (P % 16 == 0 || P == 8 || max_pages_per_seq == 1);
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
// work list is cut twice as fine as with whole-SM CTAs.  (Hc * HALVES <= 8
// also keeps every one-head box of a tile within the producer warp's lanes.)
static int choose_hc(int Hkv, int D) {
  const int cap = std::min(512 / D, 8);
  int hc = std::min(Hkv, cap);
  while (Hkv % hc != 0) --hc;
  return hc;
}

// Pipeline stages per CTA.  Two stages of 32 KB per CTA (128 KB in flight
// per SM with two CTAs) keep HBM saturated on GB300; more bytes in flight
// only lengthen the queues, which measured slower at the start and the end
// of a launch.
constexpr int kDefaultStages = 2;

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared-memory plan of the attention kernel (fused or not): kDefaultStages
// pipeline stages; if two stages do not fit, fewer kv heads go to each CTA.
// Returns false if even one head per CTA cannot have two stages.
static bool plan_attn_uncached(AttnParams& p, const DeviceInfo& dev, bool fused) {
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
            2 * align_up(4 * static_cast<size_t>(p.B), 16) + 8 * kMaxStages + 8 * (2 * kMaxStages + 5 + 8) + 48 * 4 + 256 +
            1024 /* alignment of the base */;
    stages = fixed < budget ? static_cast<int>(std::min<size_t>(kMaxStages, (budget - fixed) / p.stage_bytes)) : 0;
    if (stages >= 2 || hc == 1) break;
    int next = hc - 1;
    while (next > 1 && p.Hkv % next != 0) --next;
    hc = next;
  }
  if (stages < 2) return false;
  p.groups = p.Hkv / p.Hc;
  stages = std::min(stages, kDefaultStages);
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
  off = p.bar_off + 8 * (2 * static_cast<size_t>(stages) + 5 + 8) + 48 * 4;
  // + up to 1024 bytes that the kernel skips to align its base for the boxes
  p.smem_bytes = static_cast<int>(align_up(off, 128) + 1024);
  p.min_tiles = kMinTilesPerCta;
  return static_cast<size_t>(p.smem_bytes) <= budget;
}

static int auto_ctas_uncached(const AttnParams& p, const DeviceInfo& dev) {
  int per_sm = 0;
  if (vh::decode_attn_occupancy(p, &per_sm) != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  return std::max(1, dev.sm_count * per_sm / p.groups);
}

namespace {
// The launch-plan fields of AttnParams for one (device, shape, path, element
// type), and the automatic CTA count, computed on first use and then reused
// (the plan and the occupancy query cost more host time than the launch).
struct CachedPlan {
  bool ok;
  int auto_n;
  int fused, G, Hc, groups, stages, min_tiles, stage_bytes, q_bytes, q_row_bytes, q_tx_bytes;
  int q_off, qs_off, cum_off, len_off, pos_off, meta_off, bar_off, smem_bytes;
};
std::mutex g_plan_mu;
std::unordered_map<uint64_t, CachedPlan> g_plans;
constexpr size_t kMaxCachedPlans = 4096;

uint64_t plan_key(int dev, const AttnParams& p, bool fused) {
  // B < 2^16, Hq and Hkv <= 8192 / 1024 (checked by valid_shape: Hkv <= 1024, G <= 8), D / 64, P <= 1024
  uint64_t k = static_cast<uint64_t>(dev & 63);
  k = (k << 16) | static_cast<uint64_t>(p.B & 0xFFFF);
  k = (k << 11) | static_cast<uint64_t>(p.Hkv & 0x7FF);
  k = (k << 4) | static_cast<uint64_t>(p.Hq / p.Hkv & 0xF);
  k = (k << 2) | static_cast<uint64_t>(p.D / 64 & 0x3);
  k = (k << 11) | static_cast<uint64_t>(p.P & 0x7FF);
  k = (k << 1) | (fused ? 1u : 0u);
  k = (k << 1) | (p.f16 ? 1u : 0u);
  return k;
}
}  // namespace

bool plan_attn(AttnParams& p, const DeviceInfo& dev, bool fused, int* auto_n) {
  const uint64_t key = plan_key(dev.index, p, fused);
  CachedPlan c{};
  bool hit = false;
  {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) {
      c = it->second;
      hit = true;
    }
  }
  if (!hit) {
    AttnParams q = p;
    c.ok = plan_attn_uncached(q, dev, fused);
    c.auto_n = c.ok ? auto_ctas_uncached(q, dev) : 0;
    c.fused = q.fused;
    c.G = q.G;
    c.Hc = q.Hc;
    c.groups = q.groups;
    c.stages = q.stages;
    c.min_tiles = q.min_tiles;
    c.stage_bytes = q.stage_bytes;
    c.q_bytes = q.q_bytes;
    c.q_row_bytes = q.q_row_bytes;
    c.q_tx_bytes = q.q_tx_bytes;
    c.q_off = q.q_off;
    c.qs_off = q.qs_off;
    c.cum_off = q.cum_off;
    c.len_off = q.len_off;
    c.pos_off = q.pos_off;
    c.meta_off = q.meta_off;
    c.bar_off = q.bar_off;
    c.smem_bytes = q.smem_bytes;
    std::lock_guard<std::mutex> lk(g_plan_mu);
    if (g_plans.size() >= kMaxCachedPlans) g_plans.clear();
    g_plans[key] = c;
  }
  if (!c.ok) return false;
  p.fused = c.fused;
  p.G = c.G;
  p.Hc = c.Hc;
  p.groups = c.groups;
  p.stages = c.stages;
  p.min_tiles = c.min_tiles;
  p.stage_bytes = c.stage_bytes;
  p.q_bytes = c.q_bytes;
  p.q_row_bytes = c.q_row_bytes;
  p.q_tx_bytes = c.q_tx_bytes;
  p.q_off = c.q_off;
  p.qs_off = c.qs_off;
  p.cum_off = c.cum_off;
  p.len_off = c.len_off;
  p.pos_off = c.pos_off;
  p.meta_off = c.meta_off;
  p.bar_off = c.bar_off;
  p.smem_bytes = c.smem_bytes;
  if (auto_n) *auto_n = c.auto_n;
  return true;
}

// Fused launches that request their first stages before the dependency wait
// (VH_FLAG_PDL_KV): right after the wait, while the q rows are in flight,
// each CTA prefetches the next kL2PrefetchTiles tiles (no free stage yet) into
// L2, so the start of the stream does not wait for HBM (the kernel adds one
// more for long ranges).  One tile measured best for every range (c64 30.19
// -> 29.81 us, padded 13.41 -> 12.90 us, long 62.0 -> 61.6 us); more delay the
// q copies that gate the consumers of short ranges; the same prefetch issued
// before the wait slowed the previous kernel's end, and in launches without
// early stages (three-call attention, fused without PDL) it cost 1.2-1.4 us.
constexpr int kL2PrefetchTiles = 1;

int l2_prefetch_tiles() { return kL2PrefetchTiles; }

// Workspace: per-row split plan (int4 [B]); per-(head group, row) counters of
// the fused merge (int [Hkv][B], an upper bound on groups); partial lse
// [groups][N][2][Hq/groups] and partial outputs [...][D] (groups * Hq/groups == Hq).

int plan_rows_bytes(int B, int* len_idx, int* pos_idx) {
  const size_t c = align_up(4 * (static_cast<size_t>(B) + 1), 16), l = align_up(4 * static_cast<size_t>(B), 16);
  if (len_idx) *len_idx = static_cast<int>(c / 4);
  if (pos_idx) *pos_idx = static_cast<int>((c + l) / 4);
  return static_cast<int>(c + 2 * l);
}

WsLayout ws_layout(int B, int Hq, int Hkv, int D, int N) {
  WsLayout w;
  w.plan = 0;
  w.counters = align_up(static_cast<size_t>(B) * 16, 256);
  w.lse = w.counters + align_up(static_cast<size_t>(B) * Hkv * 4, 256);
  w.o = w.lse + align_up(static_cast<size_t>(N) * 2 * Hq * 4, 256);
  w.hdr = align_up(w.o + static_cast<size_t>(N) * 2 * Hq * D * 4, 256);
  w.rows = w.hdr + 256;
  w.recs = w.rows + align_up(static_cast<size_t>(plan_rows_bytes(B)), 256);
  w.total = w.recs + static_cast<size_t>(N) * kPlanRecInts * 4;
  return w;
}

// The driver's tensor-map encoder, looked up once through the runtime (the
// library does not link the driver library itself).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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
// 128-byte swizzle.  Full tiles: boxes of 64 elements x 16 tokens x Hc heads
// (dimension 1 = token, 2 = head), landing in shared memory as
// [head][16 tokens][128 bytes]; tiles with at most 8 live tokens: boxes of
// 64 x 8 tokens x 1 head into the first 8 rows of each head.  Token-major
// pages give dimensions 1 and 2 decreasing strides; if the encoder rejects
// that order (or VH_TMA_BOX_HEADS=1, for testing), the 8-token maps take the
// token and head dimensions in increasing stride order and every tile is
// copied as 8-token boxes (p.full_boxes = 0).  Returns false if no encoding
// is accepted.
bool encode_cache_maps(AttnParams& p) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  // L2 fill granularity of the tile reads: 256 bytes (two 128-byte box rows)
  const CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  // one pair of maps (K, V) with token and head in the given dimension order
  auto encode = [&](CUtensorMap* mk, CUtensorMap* mv, bool tok_first, cuuint32_t tokens,
                    cuuint32_t heads) -> bool {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(p.D), static_cast<cuuint64_t>(tok_first ? p.P : p.Hkv),
                                static_cast<cuuint64_t>(tok_first ? p.Hkv : p.P),
                                static_cast<cuuint64_t>(p.num_pages)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(2 * (tok_first ? p.token_stride : p.head_stride)),
                                   static_cast<cuuint64_t>(2 * (tok_first ? p.head_stride : p.token_stride)),
                                   static_cast<cuuint64_t>(2 * p.page_stride)};
    const cuuint32_t box[4] = {64, tok_first ? tokens : heads, tok_first ? heads : tokens, 1};
    for (int kv = 0; kv < 2; ++kv) {
      void* base = const_cast<uint16_t*>(kv ? p.v_cache : p.k_cache);
      if (enc(kv ? mv : mk, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    }
    return true;
  };
  // (8-token pages: every tile is two pages, copied as 8-token boxes)
  const bool forced = env_int("VH_TMA_BOX_HEADS", 0) == 1 || p.P == 8;
  if (!forced && encode(&p.tmap_k, &p.tmap_v, true, 16, static_cast<cuuint32_t>(p.Hc)) &&
      encode(&p.tmap_k8, &p.tmap_v8, true, 8, 1)) {
    p.full_boxes = 1;
    p.tm_tok_dim = 1;
    return true;
  }
  const bool tok_first = p.token_stride <= p.head_stride;
  if (!encode(&p.tmap_k8, &p.tmap_v8, tok_first, 8, 1)) return false;
  p.full_boxes = 0;
  p.tm_tok_dim = tok_first ? 1 : 2;
  return true;
}

bool too_many_tiles(int B, int max_pages_per_seq, int P) {
  const long long max_len = static_cast<long long>(max_pages_per_seq) * P;
  return max_len > (1LL << 24) || static_cast<long long>(B) * ((max_len + 15) / 16) >= (1LL << 31);
}

}  // namespace vh
