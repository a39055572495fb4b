// vh_plan.h -- launch planning of the decode kernels (internal; host side).
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "vh_kernels.h"

namespace vh {

constexpr int kMaxDevices = 64;

// Per-device facts, and the kernel attributes set once (first call on the device).
struct DeviceInfo {
  std::once_flag once;
  bool ok = false;
  int index = 0;
  int sm_count = 0;
  int smem_optin = 0;
};

// The current device's info, or null if no usable sm_103 device is current.
const DeviceInfo* device_info();

bool aligned16(const void* p);
bool valid_shape(int B, int Hq, int Hkv, int D, int P);
// Pages of a row hold whole 16-token tiles, or exactly half of one (P = 8),
// unless a row has a single page.
bool valid_paging(int P, int max_pages_per_seq);
// Without a page table, row b's pages are b * max_pages_per_seq + j: they must exist.
bool valid_table(const int32_t* page_table, int B, int max_pages_per_seq, int num_pages);
// Lengths beyond 2^24 tokens, or a tile list beyond 2^31 tiles, are not supported.
bool too_many_tiles(int B, int max_pages_per_seq, int P);
int env_int(const char* name, int dflt);

// Shared-memory plan of the attention kernel (fused or not) for p's shape and
// element type (p.B, Hq, Hkv, D, P, f16): kv heads per CTA, stages, offsets.
// False if it does not fit.  *auto_n (if given) receives the automatic CTA
// count per head group: resident CTAs per SM times the SM count.  Computed
// once per (device, shape, path, element type) and then reused.
bool plan_attn(AttnParams& p, const DeviceInfo& dev, bool fused, int* auto_n = nullptr);
// Tiles per CTA prefetched into L2 right after the dependency wait, beyond
// those the pipeline stages take first.
int l2_prefetch_tiles();

// Workspace: per-row split plan (int4 [B]); per-(head group, row) counters of
// the fused merge (int [Hkv][B], an upper bound on groups); partial lse
// [groups][N][2][Hq/groups] and partial outputs [...][D]; the per-step plan
// of vh_decode_plan (header, per-row arrays, N records).
struct WsLayout {
  size_t plan, counters, lse, o, hdr, rows, recs, total;
};
WsLayout ws_layout(int B, int Hq, int Hkv, int D, int N);
// Bytes of the per-step plan's per-row arrays: cum [B+1] | lens [B] | pos [B],
// each 16-byte aligned (the attention kernel's shared layout); *len_idx and
// *pos_idx (if given) receive the int offsets of lens and pos.
int plan_rows_bytes(int B, int* len_idx = nullptr, int* pos_idx = nullptr);

// Tensor maps of the K and V caches for the tile copies (sets p.tmap_k,
// p.tmap_v, p.tmap_k8, p.tmap_v8, p.tm_tok_dim, p.full_boxes).  False if the
// encoder rejects them.
bool encode_cache_maps(AttnParams& p);

}  // namespace vh
