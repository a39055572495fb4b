// decode_attn.cu -- paged GQA decode attention (q_len = 1), the fused decode
// step, and the LSE combine.
//
// Operation ("Engineering TTS inference in vLLM-Omni", Fish Speech S2 Pro,
// "model-specific attention kernel"): for every active row b and q head g,
// with kv head h = g / G,
//     s_j = scale * <q_rot[b,g], K[b,h,j]>,  j < L_b  (keys through the page table)
//     o   = sum_j softmax(s)_j V[b,h,j]
// with a running max (online softmax) in fp32; long rows are cut into
// segments whose partial (o, lse) are merged by the log-sum-exp recurrence.
// The fused variant also applies RoPE to q and to the new key and appends
// the new key/value to the cache ("Adding a Model", vox-serve, section 1:
// write K/V into the paged cache, then attend), and merges split rows
// itself, so one launch is one whole decode step of a layer: the CTA that
// owns a row's last tile reads the raw new k / v from the inputs, writes the
// rotated key and the value into that tile's last row in shared memory and
// into the cache slot.
//
// Design for GB300 (HBM-bound: 2-4 flops per byte of K/V):
//  * Work list.  Every active row contributes ceil(L/16) tiles of 16 tokens;
//    the list of all tiles in row order is cut into N contiguous ranges
//    that differ by at most one tile, one per CTA, on the device (each CTA
//    prefix-sums the row tile counts in shared memory).  No host sync, a static grid, and the load is
//    balanced to within one tile whatever the length mix; a row is split
//    where its tiles straddle two CTAs (at most two partial segments per CTA).
//  * Data movement.  One producer warp streams each tile into a ring of
//    shared-memory stages with tiled tensor copies (TMA, cp.async.bulk.tensor)
//    completed on an mbarrier transaction count; consumers release a stage
//    through a second mbarrier.  The cache is described to the copy engine as
//    a 4-D tensor (head_dim, token, kv head, page) whose strides come from the
//    caller, so token-major and head-major pages take the same path: per
//    64-element column block, one box of 16 tokens x all of the CTA's kv
//    heads (4 copies per tile at head_dim 128); a row's last tile with at
//    most 8 live tokens takes one-head boxes of 8 tokens instead.
//    Boxes land with the 128-byte swizzle, so ldmatrix reads of 8 rows at the
//    same column hit 8 different bank groups without padding.  In launches
//    that request their first stages before the dependency wait, the tile
//    after them is prefetched into L2 right after the wait (tensor prefetch,
//    no shared memory), so the stream's start does not wait on HBM latency
//    while the q rows arrive.  The q rows of the next segment are copied
//    (plain bulk copy) into a staging buffer while the current segment is
//    still being consumed.
//  * Math on tensor cores.  One consumer warp per kv head.  With 16 keys per
//    tile and the G q heads of the kv head padded to 8, the scores are one
//    m16n8 tile: S^T (keys x heads) = K (keys x D) . q^T, and the output is
//    O^T (D x heads) += V^T (D x keys) . P^T (keys x heads), both as
//    mma.sync m16n8k16 with operands of the cache's element type (bf16 or
//    fp16) and fp32 accumulation.  q and p are fp32 values: each is split
//    into a high part and a residual of that type (x = hi + lo to 2^-16
//    relative for bf16, 2^-22 for fp16) and both parts are multiplied, so
//    the products keep at least 16 significant bits while K and V enter
//    exactly.  P goes from the score-fragment layout to the operand
//    layout with movmatrix transposes.
//  * Stale slots (tail of the last page, slots never copied) never reach the
//    output: their scores are replaced by -inf before the max and their V rows
//    are zeroed in shared memory before the value product.
#include "vh_common.cuh"
#include "vh_kernels.h"

namespace vh {

namespace {

constexpr int kMaxHc = 8;                    // kv heads (consumer warps) per CTA
constexpr int kThreadsMax = 32 * (kMaxHc + 2);  // consumers, producer, merge warp
// Ranges of at least this many tiles prefetch one more tile into L2 right
// after the dependency wait (two in all): c64 27.90 -> 27.67 us, long 59.20 ->
// 58.65 us, padded (about 6 tiles per range) unchanged; two tiles for every
// range made padded 0.5 us slower.
constexpr int kL2LongRange = 12;

// CTA c of n takes q = T / n tiles, and the first r = T mod n CTAs one more:
// they are the first launched, so under programmatic dependent launch (CTAs
// entering as the previous kernel's leave) the extra tiles go to the CTAs
// that start streaming first.
// (The tile list has fewer than 2^31 tiles, so 32-bit arithmetic is exact.)
__device__ __forceinline__ long long range_begin(int c, int n_eff, long long T) {
  const int q = static_cast<int>(T) / n_eff, r = static_cast<int>(T) - q * n_eff;
  return static_cast<long long>(c * q + min(c, r));
}

// CTA whose range holds tile s (n_eff <= T, so q >= 1).
__device__ __forceinline__ int cta_of(long long s, int n_eff, long long T) {
  const int q = static_cast<int>(T) / n_eff, r = static_cast<int>(T) - q * n_eff;
  const int big = r * (q + 1), si = static_cast<int>(s);  // tiles of the first r CTAs
  return si < big ? si / (q + 1) : r + (si - big) / q;
}

// Page id holding tile tk of row `row`: its page (P/16 tiles per page, or
// one page of any size), or with 8-token pages (p8) page `half` of the two the
// tile spans; 0 where that page is past the row's page-table entries.  No page
// table: row b's pages are b * mps .. b * mps + mps - 1.
__device__ __forceinline__ int tile_page_id(const int32_t* page_table, int mps, bool p8, int tpp, int row, int tk,
                                            int half) {
  const int j = p8 ? 2 * tk + half : tk / tpp;
  if (j >= mps) return 0;
  const long long lp = static_cast<long long>(row) * mps + j;
  return page_table ? page_table[lp] : static_cast<int>(lp);
}

// One warp stages a segment's q rows (`bytes`, a multiple of 16) that live in
// host memory the device reads in place (VH_FLAG_HOST_IO) with plain 16-byte
// loads, then lane 0 requests the RoPE row (device memory) with a bulk copy
// whose bytes complete the phase of `bar`.  Kept out of line: the common
// path (q in device memory, bulk copies) keeps its code as it was.
__device__ __noinline__ void stage_q_host(unsigned char* dst, const uint16_t* src, int bytes, uint32_t rope_dst,
                                          const float* rope_src, int rope_bytes, uint32_t bar, int lane) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (int i = lane; i < bytes / 16; i += 32) d4[i] = s4[i];
  __syncwarp();
  if (lane == 0) {
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(rope_bytes));
    bulk_g2s(rope_dst, rope_src, static_cast<uint32_t>(rope_bytes), bar);
  }
}

// In-place inclusive prefix sum of cum[1..n] (cum[0] = 0 already).
__device__ void block_inclusive_scan(int* cum, int n, int* warp_tot) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
  const int per = (n + nthr - 1) / nthr;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int sum = 0;
  for (int i = lo; i < hi; ++i) sum += cum[1 + i];
  int x = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int v = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += y;
    }
    if (lane < nwarps) warp_tot[lane] = v;
  }
  __syncthreads();
  int run = x - sum + (warp > 0 ? warp_tot[warp - 1] : 0);
  for (int i = lo; i < hi; ++i) {
    run += cum[1 + i];
    cum[1 + i] = run;
  }
  __syncthreads();
}

enum { kMiscWarpTot = 0, kMiscAbort = 32, kMiscNVerdict = 33, kMiscVerdict = 34, kMiscInts = 48 };

// Merge the partial results of one row for the G q heads of one kv head (one
// warp): piece j comes from CTA cf + j, slot `first_slot` for j == 0 and slot
// 0 otherwise; lse in base 2.  o = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M)
// with M the running max, so each batch of U pieces costs one round trip: its
// lse and o loads are all issued before any is used (they bypass L1: other
// CTAs wrote them during this launch).
template <int D, int G, typename E>
__device__ __forceinline__ void merge_pieces(const float* __restrict__ part_lse, const float* __restrict__ part_o,
                                             long long slot_base /* (gy * N) * 2 */, int HG, int wg /* w * G */,
                                             int cf, int np, int first_slot, uint16_t* __restrict__ out_row,
                                             int lane) {
  constexpr int PER = D / 32;
  constexpr int U = 16 / G;  // pieces per batch of loads
  const float NEG_INF = __int_as_float(0xff800000);
  auto idx_of = [&](int j) -> long long {
    return (slot_base + 2LL * (cf + j) + (j == 0 ? first_slot : 0)) * HG + wg;
  };
  float M[G], o[G][PER], ws[G];
#pragma unroll
  for (int n = 0; n < G; ++n) {
    M[n] = NEG_INF;
    ws[n] = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) o[n][i] = 0.f;
  }
  for (int j0 = 0; j0 < np; j0 += U) {
    float lv[U][G], v[U][G][PER];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + u;
      const long long ix = j < np ? idx_of(j) : idx_of(j0);
#pragma unroll
      for (int n = 0; n < G; ++n) {
        lv[u][n] = j < np ? __ldcg(part_lse + ix + n) : NEG_INF;
        const float* src = part_o + (ix + n) * D + lane * PER;
        if constexpr (PER == 4) {
          const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
          v[u][n][0] = t.x;
          v[u][n][1] = t.y;
          v[u][n][2] = t.z;
          v[u][n][3] = t.w;
        } else {
          const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
          v[u][n][0] = t.x;
          v[u][n][1] = t.y;
        }
      }
    }
#pragma unroll
    for (int n = 0; n < G; ++n) {
      float mb = M[n];
#pragma unroll
      for (int u = 0; u < U; ++u) mb = fmaxf(mb, lv[u][n]);
      const float sc = exp2f(M[n] - mb);  // 0 on the first batch (M = -inf)
      ws[n] *= sc;
#pragma unroll
      for (int i = 0; i < PER; ++i) o[n][i] *= sc;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float wgt = exp2f(lv[u][n] - mb);  // 0 for the padding entries of the last batch
        ws[n] += wgt;
#pragma unroll
        for (int i = 0; i < PER; ++i) o[n][i] += wgt * v[u][n][i];
      }
      M[n] = mb;
    }
  }
#pragma unroll
  for (int n = 0; n < G; ++n) {
    const float iw = 1.f / ws[n];
    uint16_t* dst = out_row + static_cast<long long>(n) * D + lane * PER;
    if constexpr (PER == 4) {
      *reinterpret_cast<uint2*>(dst) =
          make_uint2(E::pack2(o[n][0] * iw, o[n][1] * iw), E::pack2(o[n][2] * iw, o[n][3] * iw));
    } else {
      *reinterpret_cast<uint32_t*>(dst) = E::pack2(o[n][0] * iw, o[n][1] * iw);
    }
  }
}

// Merge of a row's pieces for the fused kernel, staged through shared memory
// (used for rows of many pieces): the warp's own slices of the pipeline stages
// are free once its tile loop is done (kv head w's 2 KB rows of every
// 64-column block of K and V, of every stage: 2 * HALVES * S slices), so each
// round brings up to `nchunk / SUB` pieces (G*D*4 bytes each, SUB 2 KB copies)
// with bulk copies completed on the warp's own mbarrier, while the lanes load
// the pieces' lse values; then the round is folded into the running max / sum
// / accumulator as merge_pieces does.  One round trip per 8 pieces (4 at
// head_dim 64 or G = 8) instead of one per 16/G pieces.  The warp initialises
// its mbarrier on first use (phase 0 then).  Returns false if a wait ran out
// of time (after a second bounded wait for the copies of the round).
template <int D, int G, typename E>
__device__ __forceinline__ bool merge_pieces_staged(const float* __restrict__ part_lse,
                                                    const float* __restrict__ part_o, long long slot_base, int HG,
                                                    int wg, int cf, int np, int first_slot,
                                                    uint16_t* __restrict__ out_row, int lane, uint32_t stage0,
                                                    int stage_bytes, int S, int Hc, int w, uint32_t bar,
                                                    uint32_t& phase) {
  constexpr int PER = D / 32;
  constexpr int HALVES = D / 64;
  constexpr int PIECE = G * D * 4;                 // bytes of one piece for this warp's G heads
  constexpr int SUB = (PIECE + 2047) / 2048;       // 2 KB slices per piece
  constexpr int HPS = 2048 / (D * 4);              // heads per slice
  constexpr int PR = (2 * HALVES * 2) / SUB;       // pieces per round with two stages (upper bound)
  const float NEG_INF = __int_as_float(0xff800000);
  const int nchunk = 2 * HALVES * S;
  const int pr = min(PR, nchunk / SUB);
  auto chunk = [&](int i) -> uint32_t {
    const int st = i / (2 * HALVES), rem = i % (2 * HALVES), kv = rem / HALVES, hf = rem % HALVES;
    return stage0 + static_cast<uint32_t>(st * stage_bytes + kv * (stage_bytes / 2) + hf * Hc * 2048 + w * 2048);
  };
  auto idx_of = [&](int j) -> long long {
    return (slot_base + 2LL * (cf + j) + (j == 0 ? first_slot : 0)) * HG + wg;
  };
  float M[G], o[G][PER], ws[G];
#pragma unroll
  for (int n = 0; n < G; ++n) {
    M[n] = NEG_INF;
    ws[n] = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) o[n][i] = 0.f;
  }
  if (phase == 0u && lane == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  // the warp's slices were last read by ldmatrix and written by the tile copies
  // and the new-token patch: order those accesses before the bulk copies
  fence_proxy_async_smem();
  __syncwarp();
  for (int j0 = 0; j0 < np; j0 += pr) {
    const int nr = min(pr, np - j0);
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nr * PIECE));
    __syncwarp();
    if (lane < nr * SUB) {
      const int u = lane / SUB, sb = lane % SUB;
      const int bytes = min(2048, PIECE - sb * 2048);
      bulk_g2s(chunk(lane), part_o + idx_of(j0 + u) * D + sb * (2048 / 4), static_cast<uint32_t>(bytes), bar);
    }
    float lv[PR][G];
#pragma unroll
    for (int u = 0; u < PR; ++u) {
      const int j = j0 + u;
      const long long ix = idx_of(u < nr ? j : j0);  // (pieces past the row are not loaded)
#pragma unroll
      for (int n = 0; n < G; ++n) lv[u][n] = (u < nr) ? __ldcg(part_lse + ix + n) : NEG_INF;
    }
    const bool ok = mbar_wait(bar, phase & 1u) || mbar_wait(bar, phase & 1u);
    ++phase;
    if (!ok) return false;
#pragma unroll
    for (int n = 0; n < G; ++n) {
      float mb = M[n];
#pragma unroll
      for (int u = 0; u < PR; ++u) mb = fmaxf(mb, lv[u][n]);
      const float sc = exp2f(M[n] - mb);  // 0 on the first round (M = -inf)
      ws[n] *= sc;
#pragma unroll
      for (int i = 0; i < PER; ++i) o[n][i] *= sc;
#pragma unroll
      for (int u = 0; u < PR; ++u) {
        if (u < nr) {
          const float wgt = exp2f(lv[u][n] - mb);
          ws[n] += wgt;
          const uint32_t a = chunk(u * SUB + n / HPS) + static_cast<uint32_t>((n % HPS) * D * 4 + lane * PER * 4);
          if constexpr (PER == 4) {
            float4 t;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(t.x), "=f"(t.y), "=f"(t.z), "=f"(t.w) : "r"(a));
            o[n][0] += wgt * t.x;
            o[n][1] += wgt * t.y;
            o[n][2] += wgt * t.z;
            o[n][3] += wgt * t.w;
          } else {
            float2 t;
            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(t.x), "=f"(t.y) : "r"(a));
            o[n][0] += wgt * t.x;
            o[n][1] += wgt * t.y;
          }
        }
      }
      M[n] = mb;
    }
    // the next round's copies overwrite the slices just read
    __syncwarp();
    fence_proxy_async_smem();
  }
#pragma unroll
  for (int n = 0; n < G; ++n) {
    const float iw = 1.f / ws[n];
    uint16_t* dst = out_row + static_cast<long long>(n) * D + lane * PER;
    if constexpr (PER == 4) {
      *reinterpret_cast<uint2*>(dst) =
          make_uint2(E::pack2(o[n][0] * iw, o[n][1] * iw), E::pack2(o[n][2] * iw, o[n][3] * iw));
    } else {
      *reinterpret_cast<uint32_t*>(dst) = E::pack2(o[n][0] * iw, o[n][1] * iw);
    }
  }
  return true;
}

template <int D, int G, bool FUSED, typename E>
__global__ void __launch_bounds__(kThreadsMax, 1) decode_attn_kernel(const __grid_constant__ AttnParams p) {
  constexpr int KSTEPS = D / 16;  // k-steps of the score product = m-tiles of the value product
  constexpr int HALVES = D / 64;  // 64-element (128-byte) column blocks of a K or V row
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // the swizzled tensor copies want 1024-byte aligned boxes: every offset of
  // the plan is taken from the first 1024-byte boundary (the plan reserves it)
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hc = p.Hc, S = p.stages;
  const int c = blockIdx.x, gy = blockIdx.y;
  const int HG = Hc * G;  // q heads of this CTA
  int* cum = reinterpret_cast<int*>(smem + p.cum_off);
  int* lens = reinterpret_cast<int*>(smem + p.len_off);
  int* posv = reinterpret_cast<int*>(smem + p.pos_off);
  long long* meta = reinterpret_cast<long long*>(smem + p.meta_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  int* misc = reinterpret_cast<int*>(smem + p.bar_off + 8 * (2 * S + 5 + kMaxHc));
  volatile int* abort_flag = misc + kMiscAbort;
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + S);
  const uint32_t qfull = smem_addr(bars + 2 * S), qempty = smem_addr(bars + 2 * S + 1);
  // fused merge: consumers -> merge warp ("partial result written"), merge warp -> consumers ("counted")
  const uint32_t pready = smem_addr(bars + 2 * S + 2), mdone = smem_addr(bars + 2 * S + 3);
  const int max_len = p.max_pages_per_seq * p.P;
  // 8-token pages: a 16-token tile spans two pages (logical pages 2k and 2k + 1 of its row)
  const bool p8 = (p.P == 8);
  const uint32_t rowsbar = smem_addr(bars + 2 * S + 4);
  pdl_launch_dependents();  // the next kernel may start its CTAs as ours finish

  // ---- prologue: the work list (lengths, flags, positions and page ids are
  // read before the wait for the previous kernel: they must not be written by
  // that kernel; every other access comes after the wait) ----------------------
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, Hc);
    }
    mbar_init(qfull, 1);
    mbar_init(qempty, Hc);
    mbar_init(pready, Hc);
    mbar_init(mdone, 1);
    mbar_init(rowsbar, 1);
    fence_barrier_init();
    if (p.planned) {
      // the step's plan: its per-row arrays land in this CTA's shared arrays
      // (same layout) with one bulk copy
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(rowsbar, static_cast<uint32_t>(p.rows_bytes));
      bulk_g2s(smem_addr(cum), p.plan_rows, static_cast<uint32_t>(p.rows_bytes), rowsbar);
    }
  }
  long long T = 0, t0_pre = 0, t1_pre = 0;
  int n_eff = 0, b0_pre = 0;
  int win = 0, nxt = 0, win2 = 0, nxt2 = 0;  // producer: page ids of tiles t0 + lane, t0 + 32 + lane
  bool use_plan = false;
  if (p.planned) {
    // header and this CTA's record in the same round trip as the row arrays
    const int4 h0 = __ldcg(reinterpret_cast<const int4*>(p.plan_hdr));
    const int4 h1 = __ldcg(reinterpret_cast<const int4*>(p.plan_hdr) + 1);
    const int* rec = p.plan_recs + static_cast<long long>(c) * kPlanRecInts;
    const int4 r = __ldcg(reinterpret_cast<const int4*>(rec));
    if (warp == Hc) {
      win = __ldcg(rec + 4 + lane);
      nxt = __ldcg(rec + 4 + 32 + lane);
      if (p8) {
        win2 = __ldcg(rec + 4 + kPlanWindow + lane);
        nxt2 = __ldcg(rec + 4 + kPlanWindow + 32 + lane);
      }
    }
    // a plan made for another shape or path (or none at all) is not used
    use_plan = h0.x == kPlanMagic && h0.y == p.B && h0.z == p.N && h1.y == (FUSED ? 1 : 0) &&
               h1.z == p.max_pages_per_seq && h1.w == p.P && h0.w >= 0 && h1.x >= 0 && h1.x <= p.N &&
               (c >= h1.x || (r.x >= 0 && r.x < r.y && r.y <= h0.w && r.z >= 0 && r.z < p.B));
    T = h0.w;
    n_eff = h1.x;
    if (c < n_eff) {
      t0_pre = r.x;
      t1_pre = r.y;
      b0_pre = r.z;
    }
  }
  __syncthreads();  // barrier initialisation visible to every thread
  if (p.planned) {
    const bool landed = mbar_wait(rowsbar, 0) || mbar_wait(rowsbar, 0);
    if (__syncthreads_or(!landed)) {
      if (tid == 0) flag_error(p.err_flag, VH_ERR_TIMEOUT);
      pdl_wait();
      return;
    }
  }
  if (!use_plan) {
    // ---- no plan: tile count of every row and their prefix sum ---------------
    t0_pre = t1_pre = 0;
    b0_pre = 0;
    win = nxt = win2 = nxt2 = 0;
    for (int b = tid; b < p.B; b += blockDim.x) {
      const int a = p.active[b], L = p.seq_lens[b];
      int nt = row_tiles(a, L, max_len);
      if (a && nt == 0 && c == 0 && gy == 0) flag_error(p.err_flag, VH_ERR_SEQLEN);
      if constexpr (FUSED) {
        if (nt > 0) {
          const int pos = p.positions ? p.positions[b] : L - 1;
          if (pos < 0 || pos >= p.max_pos) {
            nt = 0;
            if (c == 0 && gy == 0) flag_error(p.err_flag, VH_ERR_POS);
          }
          posv[b] = pos;
        }
      }
      cum[1 + b] = nt;
      lens[b] = L;
    }
    if (tid == 0) cum[0] = 0;
    __syncthreads();
    block_inclusive_scan(cum, p.B, misc + kMiscWarpTot);
    T = cum[p.B];
    // (T < 2^31: 32-bit arithmetic is exact)
    n_eff = T == 0 ? 0 : min(p.N, (static_cast<int>(T) + p.min_tiles - 1) / p.min_tiles);
    // This CTA's tile range and its first row.
    t0_pre = n_eff > 0 ? range_begin(c, n_eff, T) : 0;
    t1_pre = n_eff > 0 ? range_begin(c + 1, n_eff, T) : 0;
    if (c < n_eff) {
      int lo = 0, hi = p.B - 1;  // first row with cum[b + 1] > t0
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (cum[mid + 1] > t0_pre) hi = mid; else lo = mid + 1;
      }
      b0_pre = lo;
    }
  }
  // tiles per page (P is a multiple of 16, or 8, or a row has one page of any size)
  const int tpp = (p.P + kTile - 1) / kTile;
  // row of tile tt of this CTA's range: first row with cum[row + 1] > tt
  auto row_of_from = [&](long long tt) -> int {
    int lo = b0_pre, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (cum[mid + 1] > tt) hi = mid; else lo = mid + 1;
    }
    return lo;
  };
  // page id of tile tt of this CTA's range: its page, or with 8-token pages
  // the first (half 0) or second (half 1) of its two pages; 0 past the range
  auto tile_page = [&](long long tt, int half) -> int {
    if (tt >= t1_pre) return 0;
    const int lo = row_of_from(tt);
    return tile_page_id(p.page_table, p.max_pages_per_seq, p8, tpp, lo, static_cast<int>(tt - cum[lo]), half);
  };
  if (warp == Hc && c < n_eff) {
    // The producer's first page ids are read before the wait as well.
    if (!use_plan) {
      win = tile_page(t0_pre + lane, 0);
      nxt = tile_page(t0_pre + 32 + lane, 0);
      if (p8) {
        win2 = tile_page(t0_pre + lane, 1);
        nxt2 = tile_page(t0_pre + 32 + lane, 1);
      }
    }
    // the tensor-map descriptors live in the launch parameters, not in memory
    // the previous kernel writes: fetch them before the wait as well
    if (lane == 0) prefetch_tensormap(&p.tmap_k);
    if (lane == 1) prefetch_tensormap(&p.tmap_v);
  }
  // ---- producer's box layout (used before and after the wait) --------------
  const int h0 = gy * Hc;
  // The tile's copies land at [64-column block hf][head][16 tokens][128 B] of
  // the K or V half of the stage.  Full tiles (more than 8 live tokens): one
  // box of 16 tokens x Hc heads per (K or V, hf), lanes 0 .. 2*HALVES-1.
  // Tiles with at most 8 live tokens, every tile when full_boxes == 0 and
  // every tile of 8-token pages: one box of 8 tokens x 1 head per (K or V, hf,
  // head, 8-token group), lane (((group * Hc + head) * HALVES + hf) * 2 + kv);
  // with 8-token pages, group g is token 0.. of the tile's page g.
  const int l_kv = lane & 1, l_hf = (lane >> 1) % HALVES;
  const int l_head = (lane / (2 * HALVES)) % Hc, l_g = lane / (2 * HALVES * Hc);
  const void* l_map16 = l_kv ? static_cast<const void*>(&p.tmap_v) : static_cast<const void*>(&p.tmap_k);
  const void* l_map8 = l_kv ? static_cast<const void*>(&p.tmap_v8) : static_cast<const void*>(&p.tmap_k8);
  const uint32_t l_off16 = static_cast<uint32_t>(l_kv * (p.stage_bytes / 2) + l_hf * Hc * 2048);
  const uint32_t l_off8 = l_off16 + static_cast<uint32_t>(l_head * 2048 + l_g * 1024);
  // Tile state of the producer: stage ring position and, for tile t of row
  // b, its box coordinates, the append slot and the bytes its boxes deliver.
  int npre = 0;  // tiles whose boxes were requested before the wait
  // K/V tiles are read once per launch: copied with the L2 evict-first
  // policy, so the stream does not push out what is read again (q rows, RoPE
  // rows, page ids, partial results; c64 29.32 -> 27.89 us, long 61.07 ->
  // 59.16 us, padded 12.96 -> 12.73 us in one A/B call)
  const uint64_t kv_policy = l2_policy_evict_first();
  auto issue_tile = [&](long long t, int b, long long rt0, long long rt1, int tin_page, int page, bool page_ok,
                        int page2, bool page2_ok, int stage) {
    const int tok0 = static_cast<int>(t - rt0) * kTile;
    const int nvalid = min(kTile, lens[b] - tok0);
    const bool last_of_row = (t == rt1 - 1);
    const int tokc = tin_page * kTile;
    const bool two_groups = nvalid > 8;
    const uint32_t st = smem_addr(smem) + static_cast<uint32_t>(stage) * p.stage_bytes;
    long long meta_val = -1;
    if constexpr (FUSED) {
      // the new token's cache slot: slot nvalid - 1 of the tile (with 8-token
      // pages, in the tile's second page if it is past the first 8 tokens)
      const int sl = nvalid - 1;
      const bool second = p8 && sl >= 8;
      if (last_of_row && (second ? page2_ok : page_ok))
        meta_val = static_cast<long long>(second ? page2 : page) * p.page_stride +
                   static_cast<long long>(second ? sl - 8 : tokc + sl) * p.token_stride +
                   static_cast<long long>(h0) * p.head_stride;
    }
    // bytes of the boxes issued: both token groups, or the first only
    const uint32_t tx = static_cast<uint32_t>(two_groups ? p.stage_bytes : p.stage_bytes / 2);
    const uint32_t fb = full0 + 8 * stage;
    if (lane == 0) {
      if constexpr (FUSED) meta[stage] = meta_val;
      mbar_arrive_expect_tx(fb, tx);
    }
    __syncwarp();
    if (two_groups && p.full_boxes && !p8) {
      if (lane < 2 * HALVES) tma_load_4d_hint(st + l_off16, l_map16, l_hf * 64, tokc, h0, page, fb, kv_policy);
    } else if (lane < 2 * HALVES * Hc * (two_groups ? 2 : 1)) {
      const int tk = p8 ? 0 : tokc + 8 * l_g;
      const int c1 = p.tm_tok_dim == 1 ? tk : h0 + l_head, c2 = p.tm_tok_dim == 1 ? h0 + l_head : tk;
      tma_load_4d_hint(st + l_off8, l_map8, l_hf * 64, c1, c2, (p8 && l_g) ? page2 : page, fb, kv_policy);
    }
  };
  // L2 prefetch (no shared memory, no completion) of this CTA's tiles [ta, tb),
  // tb - t0 <= 32 (page ids from the first window)
  auto prefetch_l2 = [&](long long ta, long long tb) {
    int b = row_of_from(ta);
    long long rt1 = cum[b + 1];
    for (long long t = ta; t < tb; ++t) {
      while (t >= rt1) rt1 = cum[++b + 1];
      const long long rt0 = cum[b];
      const int page = __shfl_sync(0xffffffffu, win, static_cast<int>(t - t0_pre));
      const int page2 = p8 ? __shfl_sync(0xffffffffu, win2, static_cast<int>(t - t0_pre)) : 0;
      const int nvalid = min(kTile, lens[b] - static_cast<int>(t - rt0) * kTile);
      const int tokc = (static_cast<int>(t - rt0) % tpp) * kTile;
      const int pg = (p8 && l_g) ? page2 : page;
      if (nvalid > 8 && p.full_boxes && !p8) {
        if (lane < 2 * HALVES && page >= 0 && page < p.num_pages)
          tma_prefetch_l2_4d(l_map16, l_hf * 64, tokc, h0, page);
      } else if (lane < 2 * HALVES * Hc * (nvalid > 8 ? 2 : 1) && pg >= 0 && pg < p.num_pages) {
        // (bad page ids are skipped here and flagged when the tile is copied)
        const int tk = p8 ? 0 : tokc + 8 * l_g;
        const int c1 = p.tm_tok_dim == 1 ? tk : h0 + l_head, c2 = p.tm_tok_dim == 1 ? h0 + l_head : tk;
        tma_prefetch_l2_4d(l_map8, l_hf * 64, c1, c2, pg);
      }
    }
  };
  if (FUSED && p.prefetch_kv && warp == Hc && c < n_eff) {
    // The cached K/V of this call are not written by the previous kernel
    // (the caller's promise with VH_FLAG_PDL_KV), and the new token's row is
    // rewritten from v_new / the rotated k_new after the wait: the first
    // stages can be requested before the wait.
    int b = b0_pre;
    long long rt1 = cum[b + 1];
    const long long n = min(static_cast<long long>(S), t1_pre - t0_pre);
    for (long long t = t0_pre; t < t0_pre + n; ++t) {
      while (t >= rt1) rt1 = cum[++b + 1];
      const long long rt0 = cum[b];
      const int tin_page = static_cast<int>(t - rt0) % tpp;
      int page = __shfl_sync(0xffffffffu, win, static_cast<int>(t - t0_pre));
      int page2 = p8 ? __shfl_sync(0xffffffffu, win2, static_cast<int>(t - t0_pre)) : 0;
      const bool page_ok = page >= 0 && page < p.num_pages;
      const bool page2_ok = page2 >= 0 && page2 < p.num_pages;
      if (!page_ok) page = 0;  // flagged again after the wait
      if (!page2_ok) page2 = 0;
      issue_tile(t, b, rt0, rt1, tin_page, page, page_ok, page2, page2_ok, static_cast<int>(t - t0_pre));
      ++npre;
    }
  }
  // The first segment's q rows (and, fused, its RoPE row) are requested at
  // once: the consumers cannot start before they arrive, and the producer may
  // still be busy with the requests it makes before the wait (page ids, first
  // stages).  Later segments' q rows come from the producer.  q in host
  // memory (VH_FLAG_HOST_IO) is written by the host before the launch, never
  // by the previous kernel, so consumer warp 0 loads those rows before the
  // wait (end-to-end c64 step 29.43 -> 28.41 us in one A/B call); q in device
  // memory may come from the previous kernel and is requested by thread 0 as
  // soon as the wait returns.
  const bool early_q = p.early_q && c < n_eff;
  if (FUSED && p.host_io && early_q && warp == 0) {
    const long long qrow = static_cast<long long>(b0_pre) * p.Hq + static_cast<long long>(h0) * G;
    stage_q_host(smem + p.q_off, p.q + qrow * D, HG * D * 2, smem_addr(smem + p.q_off) + HG * p.q_row_bytes,
                 p.cos_sin + static_cast<long long>(posv[b0_pre]) * D, p.q_tx_bytes, qfull, lane);
  }
  pdl_wait();

  if (!(FUSED && p.host_io) && early_q && tid == 0) {
    mbar_arrive_expect_tx(qfull, static_cast<uint32_t>(p.q_tx_bytes));
    const long long qrow = static_cast<long long>(b0_pre) * p.Hq + static_cast<long long>(h0) * G;
    const uint32_t qdst = smem_addr(smem + p.q_off);
    if constexpr (FUSED) {
      bulk_g2s(qdst, p.q + qrow * D, HG * D * 2, qfull);
      bulk_g2s(qdst + HG * p.q_row_bytes, p.cos_sin + static_cast<long long>(posv[b0_pre]) * D, D * 4, qfull);
    } else {
      bulk_g2s(qdst, p.q_rot + qrow * D, HG * D * 4, qfull);
    }
  }

  // ---- per-row duties, rows b = c (mod N): split plan, zero padding rows ---
  for (int b = c; b < p.B; b += p.N) {
    const int nt = cum[b + 1] - cum[b];
    if (nt == 0) {
      uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<long long>(b) * p.Hq + gy * HG) * D);
      for (int i = tid; i < HG * D / 8; i += blockDim.x) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      if (!FUSED && gy == 0 && tid == 0) p.plan[b] = make_int4(-1, -1, 0, 0);
    } else if (!FUSED && gy == 0 && tid == 0) {
      const long long s0 = cum[b], s1 = cum[b + 1] - 1;
      const int cf = cta_of(s0, n_eff, T), cl = cta_of(s1, n_eff, T);
      p.plan[b] = make_int4(cf, cl, range_begin(cf, n_eff, T) == s0 ? 0 : 1, nt);
    }
  }
  if (c >= n_eff) return;
  const long long t0 = t0_pre, t1 = t1_pre;
  const int b0 = b0_pre;

  if (FUSED && warp == Hc + 1) {
    // ======================= merge warp (fused) ============================
    // Counts this CTA's partial results per row, off the streaming path: the
    // consumers only signal that a partial result is written.  A CTA has at
    // most two partial segments: its first row, if it started or stops inside
    // it, and its last row, if that is another row and stops inside it.
    int b_last;
    {
      int lo = b0, hi = p.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (cum[mid + 1] > t1 - 1) hi = mid; else lo = mid + 1;
      }
      b_last = lo;
    }
    int rows[2], n = 0;
    if (t0 > cum[b0] || t1 < cum[b0 + 1]) rows[n++] = b0;
    if (b_last != b0 && t1 < cum[b_last + 1]) rows[n++] = b_last;
    int done = 0;
    for (int k = 0; k < n; ++k) {
      if (!mbar_wait(pready, k & 1)) {
        if (lane == 0) flag_error(p.err_flag, VH_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      if (lane == 0) {
        const int rb = rows[k];
        const long long s0 = cum[rb], s1 = cum[rb + 1] - 1;
        const int cf = cta_of(s0, n_eff, T), cl = cta_of(s1, n_eff, T);
        // acquire-release at GPU scope: publishes the consumers' partial writes
        // (ordered before it by the stage barrier) and, for the last arrival,
        // makes every other piece visible to the merge that follows
        int* counter = p.counters + static_cast<long long>(gy) * p.B + rb;
        const int old = atom_add_acq_rel_gpu(counter, 1);
        const int last = (old == cl - cf);
        if (last) *counter = 0;  // every piece has arrived: ready for the next call
        int* v = misc + kMiscVerdict + 5 * k;
        v[0] = last;
        v[1] = rb;
        v[2] = cf;
        v[3] = cl;
        v[4] = range_begin(cf, n_eff, T) == s0 ? 0 : 1;
      }
      ++done;
    }
    if (lane == 0) {
      misc[kMiscNVerdict] = done;
      mbar_arrive(mdone);
    }
    return;
  }

  if (warp == Hc) {
    // ======================= producer warp =================================
    // Everything a tile needs is computed before the wait for its stage, so
    // that a released stage is refilled at once: the row walk is incremental,
    // and the page ids come from a 32-tile window that is loaded (one
    // coalesced load per lane) a whole window ahead of its use.
    long long wb = t0;
    int b = b0;
    long long rt0 = cum[b], rt1 = cum[b + 1];
    int tin_page = static_cast<int>(t0 - rt0) % tpp;  // tile index within its page
    int stage = 0, round = 0, nseg = 0;
    long long issued = 0;
    bool aborted = false;
    for (long long t = t0; t < t1; ++t, ++issued) {
      bool new_seg = (t == t0);
      if (t > t0 && ++tin_page == tpp) tin_page = 0;
      while (t >= rt1) {
        ++b;
        rt0 = rt1;
        rt1 = cum[b + 1];
        new_seg = true;
        tin_page = 0;
      }
      if (t == wb + 32) {
        wb += 32;
        win = nxt;
        nxt = tile_page(wb + 32 + lane, 0);
        if (p8) {
          win2 = nxt2;
          nxt2 = tile_page(wb + 32 + lane, 1);
        }
      }
      int page = __shfl_sync(0xffffffffu, win, static_cast<int>(t - wb));
      const bool page_ok = page >= 0 && page < p.num_pages;
      if (!page_ok) {
        if (lane == 0) flag_error(p.err_flag, VH_ERR_PAGE);
        page = 0;
      }
      // 8-token pages: the tile's second page, read only when the tile has more than 8 live tokens
      int page2 = p8 ? __shfl_sync(0xffffffffu, win2, static_cast<int>(t - wb)) : 0;
      const bool page2_ok = page2 >= 0 && page2 < p.num_pages;
      if (!page2_ok) {
        if (p8 && lane == 0 && lens[b] - static_cast<int>(t - rt0) * kTile > 8) flag_error(p.err_flag, VH_ERR_PAGE);
        page2 = 0;
      }
      if (new_seg) {
        // q rows of this segment's row (fused: 16-bit q and the RoPE row of its
        // position) into the staging buffer, once the consumers have taken
        // the previous segment's q into registers.
        if (nseg > 0 && !mbar_wait(qempty, (nseg - 1) & 1)) {
          if (lane == 0) flag_error(p.err_flag, VH_ERR_TIMEOUT);
          *abort_flag = 1;
          aborted = true;
          break;
        }
        if (FUSED && p.host_io && !(nseg == 0 && early_q)) {
          // q in host memory: the producer loads the rows itself (plain loads)
          const long long qrow = static_cast<long long>(b) * p.Hq + static_cast<long long>(h0) * G;
          stage_q_host(smem + p.q_off, p.q + qrow * D, HG * D * 2, smem_addr(smem + p.q_off) + HG * p.q_row_bytes,
                       p.cos_sin + static_cast<long long>(posv[b]) * D, p.q_tx_bytes, qfull, lane);
        } else if (lane == 0 && !(nseg == 0 && early_q)) {
          // the q rows of the segment's row (one contiguous copy) and, fused, the RoPE row
          mbar_arrive_expect_tx(qfull, static_cast<uint32_t>(p.q_tx_bytes));
          const long long qrow = static_cast<long long>(b) * p.Hq + static_cast<long long>(h0) * G;
          const uint32_t qdst = smem_addr(smem + p.q_off);
          if constexpr (FUSED) {
            bulk_g2s(qdst, p.q + qrow * D, HG * D * 2, qfull);
            bulk_g2s(qdst + HG * p.q_row_bytes, p.cos_sin + static_cast<long long>(posv[b]) * D, D * 4, qfull);
          } else {
            bulk_g2s(qdst, p.q_rot + qrow * D, HG * D * 4, qfull);
          }
        }
        ++nseg;
        if (t == t0 && p.l2_tiles > 0) {
          // while the q rows and the first stages arrive, the next tiles
          // (which have no free stage yet) are read into L2: one more for
          // ranges of at least kL2LongRange tiles
          const long long ta = t0 + S;
          const int n_l2 = p.l2_tiles + (t1 - t0 >= kL2LongRange ? 1 : 0);
          prefetch_l2(ta, min(t1, min(t0 + 32, ta + n_l2)));
        }
      }
      // the boxes of this tile (the new token's row arrives as whatever the
      // cache slot holds; the consumers overwrite it with the rotated key and
      // v_new), unless they were requested before the wait
      if (issued >= npre) {
        if (issued >= S && !mbar_wait(empty0 + 8 * stage, (round - 1) & 1)) {
          if (lane == 0) flag_error(p.err_flag, VH_ERR_TIMEOUT);
          *abort_flag = 1;
          aborted = true;
          break;
        }
        if (*abort_flag) {
          aborted = true;
          break;
        }
        issue_tile(t, b, rt0, rt1, tin_page, page, page_ok, page2, page2_ok, stage);
      }
      if (++stage == S) {
        stage = 0;
        ++round;
      }
    }
    if (aborted) {
      // Let the copies already issued land before the CTA's shared memory goes away
      // (including those requested before the wait).
      const long long req = max(issued, static_cast<long long>(npre));
      const long long n = min(req, static_cast<long long>(S));
      for (long long k = req - n; k < req; ++k)
        (void)mbar_wait(full0 + 8 * static_cast<int>(k % S), static_cast<uint32_t>((k / S) & 1));
      if (nseg > 0) (void)mbar_wait(qfull, (nseg - 1) & 1);
    }
    return;
  }

  // ========================= consumer warps ==================================
  const int w = warp;            // kv head within the CTA
  const int h = gy * Hc + w;     // kv head
  const int g4 = lane >> 2, t4 = lane & 3;  // mma fragment coordinates
  const float NEG_INF = __int_as_float(0xff800000);
  // ldmatrix row (key) and 16-byte column chunk of this lane: K tile (keys x
  // dims; k-step k reads chunk 2k + (lane >> 4)) and V tile (read transposed;
  // m-tile mt reads chunk 2 mt + ((lane >> 3) & 1)).  In the swizzled boxes,
  // chunk c of row r sits at chunk c ^ (r & 7); as 2k is even, the physical
  // chunk is (2k mod 8) ^ ksw with ksw = (lane >> 4) ^ (r & 7).
  const int ka_row = (lane & 7) + 8 * ((lane >> 3) & 1);
  const int va_row = (lane & 7) + 8 * (lane >> 4);
  const int ksw = (lane >> 4) ^ (ka_row & 7), vsw = ((lane >> 3) & 1) ^ (va_row & 7);
  // Stage layout of K (and then V): [64-column block][head][16 tokens][128 B];
  // row r of head w of a column block is at row_off(r).
  const uint32_t half_bytes = static_cast<uint32_t>(Hc) * 2048u;  // one 64-column block of all heads
  auto row_off = [&](int r) -> uint32_t { return static_cast<uint32_t>(w * 2048 + r * 128); };
  const uint32_t k_lane = row_off(ka_row);
  const uint32_t v_lane = static_cast<uint32_t>(p.stage_bytes / 2) + row_off(va_row);

  // fused: per-lane RMSNorm weights (q: the lane's fixed elements in step (1) of
  // the fragment build; k: the lane's pairs in the append patch)
  constexpr int NQU = D / 4;              // 4-element units per q head (32 or 16)
  constexpr int KPAIRS = (D / 2 + 31) / 32;
  float wq[4] = {1.f, 1.f, 1.f, 1.f}, wk[2 * KPAIRS];
#pragma unroll
  for (int j = 0; j < 2 * KPAIRS; ++j) wk[j] = 1.f;
  // weights in the order (x0, x1, y0, y1) of the rotation pairs (x, y): pair i is
  // (i, i + D/2), or (2i, 2i + 1) with interleaved RoPE
  const bool ilv = p.rope_interleaved != 0;
  if constexpr (FUSED) {
    const int iq = 2 * (lane % NQU);
    if (p.q_norm_w) {
      if (ilv) {
        const float4 a = *reinterpret_cast<const float4*>(p.q_norm_w + 2 * iq);
        wq[0] = a.x;
        wq[1] = a.z;
        wq[2] = a.y;
        wq[3] = a.w;
      } else {
        const float2 a = *reinterpret_cast<const float2*>(p.q_norm_w + iq);
        const float2 c2 = *reinterpret_cast<const float2*>(p.q_norm_w + D / 2 + iq);
        wq[0] = a.x;
        wq[1] = a.y;
        wq[2] = c2.x;
        wq[3] = c2.y;
      }
    }
    if (p.k_norm_w) {
#pragma unroll
      for (int j = 0; j < KPAIRS; ++j) {
        const int i = lane + 32 * j;
        if (i < D / 2) {
          wk[2 * j] = p.k_norm_w[ilv ? 2 * i : i];
          wk[2 * j + 1] = p.k_norm_w[ilv ? 2 * i + 1 : i + D / 2];
        }
      }
    }
  }
  (void)wq;
  (void)wk;

  uint32_t qh[KSTEPS][2], ql[KSTEPS][2];  // q^T operand fragments (high / residual parts)
  float acc[KSTEPS][4];                   // O^T fragments: dims mt*16 + g4 (+8), heads 2 t4 (+1)
  float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
  float rc[(D / 2 + 31) / 32], rs[(D / 2 + 31) / 32];  // fused: RoPE row for the new key
  // fused: the new token's raw key (pair j of this lane: first element in the
  // low half, partner in the high half) and this lane's 16 bytes of v_new,
  // loaded when a segment that holds the row's last tile starts
  uint32_t knew[KPAIRS];
  uint4 vnew = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int j = 0; j < KPAIRS; ++j) knew[j] = 0u;
  (void)rc;
  (void)rs;
  (void)knew;
  (void)vnew;

  int b = b0;
  long long rt0 = cum[b], rt1 = cum[b + 1];
  int seg = 0, nseg = 0, stage = 0, round = 0, npart = 0;
  for (long long t = t0; t < t1; ++t) {
    bool new_seg = (t == t0), new_row = false;
    while (t >= rt1) {
      ++b;
      rt0 = rt1;
      rt1 = cum[b + 1];
      new_row = true;
      new_seg = true;
    }
    if (new_row) ++seg;
    const long long sb = max(t0, rt0), se = min(t1, rt1);

    if (new_seg) {
      if (!mbar_wait(qfull, nseg & 1)) {
        if (lane == 0) flag_error(p.err_flag, VH_ERR_TIMEOUT);
        *abort_flag = 1;
        return;
      }
      const unsigned char* qb = smem + p.q_off;
      const float* cs = reinterpret_cast<const float*>(qb + HG * p.q_row_bytes);  // fused: RoPE row
      // fused: (1) all 32 lanes rotate this warp's G q rows (RoPE in fp32, pairs
      // (i, i + D/2), or (2i, 2i + 1) interleaved) into padded per-warp fp32 rows
      // (D*4 + 32 bytes) so that (2) every lane reads its operand pairs without
      // bank conflicts.
      // Three-call path: the staged rows are fp32 already and are read directly.
      constexpr int QS_ROW = D * 4 + 32;
      const unsigned char* qsrc;
      int qstride;
      if constexpr (FUSED) {
        unsigned char* qs = smem + p.qs_off + w * G * QS_ROW;
        // every lane runs each round (the per-head RMS reduction shuffles)
        for (int e0 = 0; e0 < G * NQU; e0 += 32) {
          const int e = e0 + lane;
          const bool valid = e < G * NQU;
          const int n = valid ? e / NQU : 0;
          const int i = (e % NQU) * 2;  // i, i+1 in [0, D/2)
          const unsigned char* row = qb + (w * G + n) * p.q_row_bytes;
          // xv: first elements of pairs i and i + 1, yv: their partners
          float2 xv = make_float2(0.f, 0.f), yv = make_float2(0.f, 0.f);
          if (valid) {
            if (ilv) {
              const uint2 w2 = *reinterpret_cast<const uint2*>(row + 4 * i);  // elements 2i .. 2i+3
              const float2 a = E::to_float2(w2.x), c2 = E::to_float2(w2.y);
              xv = make_float2(a.x, c2.x);
              yv = make_float2(a.y, c2.y);
            } else {
              xv = E::to_float2(*reinterpret_cast<const uint32_t*>(row + 2 * i));
              yv = E::to_float2(*reinterpret_cast<const uint32_t*>(row + 2 * (i + D / 2)));
            }
          }
          if (p.q_norm_w) {
            // RMSNorm in fp32: the NQU lanes of a head hold its D elements
            float ss = xv.x * xv.x + xv.y * xv.y + yv.x * yv.x + yv.y * yv.y;
#pragma unroll
            for (int off = 1; off < NQU; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float r = rsqrtf(ss / static_cast<float>(D) + p.norm_eps);
            xv = make_float2(wq[0] * (xv.x * r), wq[1] * (xv.y * r));
            yv = make_float2(wq[2] * (yv.x * r), wq[3] * (yv.y * r));
          }
          if (valid) {
            const float2 cv = *reinterpret_cast<const float2*>(cs + i);
            const float2 sv = *reinterpret_cast<const float2*>(cs + D / 2 + i);
            float* dst = reinterpret_cast<float*>(qs + n * QS_ROW);
            const float2 rx = make_float2(xv.x * cv.x - yv.x * sv.x, xv.y * cv.y - yv.y * sv.y);
            const float2 ry = make_float2(yv.x * cv.x + xv.x * sv.x, yv.y * cv.y + xv.y * sv.y);
            if (ilv) {
              *reinterpret_cast<float4*>(dst + 2 * i) = make_float4(rx.x, ry.x, rx.y, ry.y);
            } else {
              *reinterpret_cast<float2*>(dst + i) = rx;
              *reinterpret_cast<float2*>(dst + i + D / 2) = ry;
            }
          }
        }
        __syncwarp();
        qsrc = qs;
        qstride = QS_ROW;
      } else {
        qsrc = qb + w * G * p.q_row_bytes;
        qstride = p.q_row_bytes;
      }
      // (2) each lane takes its operand pairs: head g4, dims 16k + 2 t4 (+1) and +8 (+9)
      const int n = g4;
      const float* qrow = reinterpret_cast<const float*>(qsrc + (n < G ? n : 0) * qstride);
#pragma unroll
      for (int k = 0; k < KSTEPS; ++k) {
        float2 a = make_float2(0.f, 0.f), c2 = make_float2(0.f, 0.f);
        if (n < G) {
          a = *reinterpret_cast<const float2*>(qrow + 16 * k + 2 * t4);
          c2 = *reinterpret_cast<const float2*>(qrow + 16 * k + 2 * t4 + 8);
        }
        split2<E>(a.x, a.y, qh[k][0], ql[k][0]);
        split2<E>(c2.x, c2.y, qh[k][1], ql[k][1]);
      }
      if constexpr (FUSED) {
#pragma unroll
        for (int j = 0; j < (D / 2 + 31) / 32; ++j) {
          const int i = lane + 32 * j;
          rc[j] = i < D / 2 ? cs[i] : 0.f;
          rs[j] = i < D / 2 ? cs[D / 2 + i] : 0.f;
        }
        if (se == rt1) {
          // this segment ends the row: fetch the new key and value now, used at its last tile
          const uint16_t* kn = p.k_new + (static_cast<long long>(b) * p.Hkv + h) * D;
#pragma unroll
          for (int j = 0; j < KPAIRS; ++j) {
            const int i = lane + 32 * j;
            if (i < D / 2)
              knew[j] = ilv ? *reinterpret_cast<const uint32_t*>(kn + 2 * i)
                            : static_cast<uint32_t>(kn[i]) | (static_cast<uint32_t>(kn[i + D / 2]) << 16);
          }
          if (lane < D / 8)
            vnew = *reinterpret_cast<const uint4*>(p.v_new + (static_cast<long long>(b) * p.Hkv + h) * D + lane * 8);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty);
      ++nseg;
      m0 = m1 = NEG_INF;
      l0 = l1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    }

    const int tok0 = static_cast<int>(t - rt0) * kTile;
    const int nvalid = min(kTile, lens[b] - tok0);
    if (!mbar_wait(full0 + 8 * stage, round & 1)) {
      if (lane == 0) flag_error(p.err_flag, VH_ERR_TIMEOUT);
      *abort_flag = 1;
      return;
    }
    // this stage: K boxes [D/64][Hc][16][128 B], then V boxes, all swizzled
    unsigned char* stg = smem + static_cast<long long>(stage) * p.stage_bytes;
    unsigned char* vst = stg + p.stage_bytes / 2;
    bool touched = false;

    if constexpr (FUSED) {
      if (t == rt1 - 1) {
        // the new token (row nvalid-1 of the tile, which the box copy filled
        // with whatever the cache slot held): (RMSNorm and) rotate its key,
        // write key and value into the tile row and append them to the cache
        const int rr = nvalid - 1;
        unsigned char* krow = stg + row_off(rr);   // + column block * half_bytes
        unsigned char* vrow = vst + row_off(rr);
        // byte offset of element e of row rr within this head's boxes
        auto elem_off = [&](int e) -> uint32_t {
          return static_cast<uint32_t>(e >> 6) * half_bytes + (((((e >> 3) & 7) ^ (rr & 7))) << 4) + (e & 7) * 2;
        };
        const long long dst = meta[stage];
        float kx[KPAIRS], ky[KPAIRS];
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < KPAIRS; ++j) {
          const float2 xy = E::to_float2(knew[j]);  // zero for lanes without a pair
          kx[j] = xy.x;
          ky[j] = xy.y;
          ss += kx[j] * kx[j] + ky[j] * ky[j];
        }
        if (p.k_norm_w) {
          // RMSNorm of the new key in fp32 (the warp holds its D elements)
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
          const float r = rsqrtf(ss / static_cast<float>(D) + p.norm_eps);
#pragma unroll
          for (int j = 0; j < KPAIRS; ++j) {
            kx[j] = wk[2 * j] * (kx[j] * r);
            ky[j] = wk[2 * j + 1] * (ky[j] * r);
          }
        }
#pragma unroll
        for (int j = 0; j < KPAIRS; ++j) {
          const int i = lane + 32 * j;
          if (i < D / 2) {
            const float x = kx[j], y = ky[j];
            const float xr = x * rc[j] - y * rs[j], yr = y * rc[j] + x * rs[j];
            uint16_t* cache_row = p.k_cache_w + dst + static_cast<long long>(w) * p.head_stride;
            if (ilv) {
              const uint32_t xy = E::pack2(xr, yr);
              *reinterpret_cast<uint32_t*>(krow + elem_off(2 * i)) = xy;
              if (dst >= 0) *reinterpret_cast<uint32_t*>(cache_row + 2 * i) = xy;
            } else {
              const uint16_t xb = E::bits(xr), yb = E::bits(yr);
              *reinterpret_cast<uint16_t*>(krow + elem_off(i)) = xb;
              *reinterpret_cast<uint16_t*>(krow + elem_off(i + D / 2)) = yb;
              if (dst >= 0) {
                cache_row[i] = xb;
                cache_row[i + D / 2] = yb;
              }
            }
          }
        }
        if (lane < D / 8) {
          *reinterpret_cast<uint4*>(vrow + elem_off(lane * 8)) = vnew;
          if (dst >= 0)
            *reinterpret_cast<uint4*>(p.v_cache_w + dst + static_cast<long long>(w) * p.head_stride + lane * 8) = vnew;
        }
        touched = true;
      }
    }
    if (nvalid < kTile) {
      // stale V rows would meet p = 0 in the product; make them exact zeros
      // (whole rows, so the swizzle does not matter)
      constexpr int CH = D / 8;  // 16-byte chunks per row, over the column blocks
      for (int r = nvalid + lane / CH; r < kTile; r += 32 / CH) {
        const int ch = lane % CH;
        *reinterpret_cast<uint4*>(vst + (ch >> 3) * half_bytes + row_off(r) + (ch & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      touched = true;
    }
    if (touched) __syncwarp();

    // ---- scores S^T = K q^T on tensor cores ----------------------------------
    float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const uint32_t ka = smem_addr(stg) + k_lane;
#pragma unroll
      for (int k = 0; k < KSTEPS; ++k) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(ka + (k >> 2) * half_bytes + ((((2 * k) & 7) ^ ksw) << 4), a0, a1, a2, a3);
        E::mma(sh, a0, a1, a2, a3, qh[k][0], qh[k][1]);
        E::mma(sl, a0, a1, a2, a3, ql[k][0], ql[k][1]);
      }
    }
    // lane holds keys g4 (s[0], s[1]) and g4 + 8 (s[2], s[3]), heads 2 t4 and 2 t4 + 1
    const bool va = g4 < nvalid, vb = g4 + 8 < nvalid;
    const float s0 = va ? (sh[0] + sl[0]) * p.scale_log2 : NEG_INF;
    const float s1 = va ? (sh[1] + sl[1]) * p.scale_log2 : NEG_INF;
    const float s2 = vb ? (sh[2] + sl[2]) * p.scale_log2 : NEG_INF;
    const float s3 = vb ? (sh[3] + sl[3]) * p.scale_log2 : NEG_INF;

    // ---- online softmax (per head; reduce over the 8 lanes sharing t4) -------
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    const float p0 = exp2f(s0 - mn0), p2 = exp2f(s2 - mn0);
    const float p1 = exp2f(s1 - mn1), p3 = exp2f(s3 - mn1);
    l0 = l0 * al0 + (p0 + p2);
    l1 = l1 * al1 + (p1 + p3);
    m0 = mn0;
    m1 = mn1;
    uint32_t ph01, pl01, ph23, pl23;
    split2<E>(p0, p1, ph01, pl01);
    split2<E>(p2, p3, ph23, pl23);
    const uint32_t bh0 = movm_t(ph01), bh1 = movm_t(ph23);
    const uint32_t bl0 = movm_t(pl01), bl1 = movm_t(pl23);
    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        acc[mt][0] *= al0;
        acc[mt][1] *= al1;
        acc[mt][2] *= al0;
        acc[mt][3] *= al1;
      }
    }

    // ---- values O^T += V^T P^T on tensor cores ---------------------------------
    {
      const uint32_t vaddr = smem_addr(stg) + v_lane;
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vaddr + (mt >> 2) * half_bytes + ((((2 * mt) & 7) ^ vsw) << 4), a0, a1, a2, a3);
        E::mma(acc[mt], a0, a1, a2, a3, bh0, bh1);
        E::mma(acc[mt], a0, a1, a2, a3, bl0, bl1);
      }
    }
    if (touched) fence_proxy_async_smem();  // generic writes before the next bulk copy into this stage
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * stage);
    if (++stage == S) {
      stage = 0;
      ++round;
    }

    // ---- end of a segment: finished row or partial result ----------------------
    if (t == se - 1) {
      float L0 = l0, L1 = l1;
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        L0 += __shfl_xor_sync(0xffffffffu, L0, off);
        L1 += __shfl_xor_sync(0xffffffffu, L1, off);
      }
      const float il0 = 1.f / L0, il1 = 1.f / L1;
      const int n0 = 2 * t4, n1 = 2 * t4 + 1;
      const bool full_row = (sb == rt0) && (se == rt1);
      if (full_row) {
        uint16_t* o0 = p.out + (static_cast<long long>(b) * p.Hq + static_cast<long long>(h) * G + n0) * D;
        uint16_t* o1 = o0 + D;
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
          const int d = mt * 16 + g4;
          if (n0 < G) {
            o0[d] = E::bits(acc[mt][0] * il0);
            o0[d + 8] = E::bits(acc[mt][2] * il0);
          }
          if (n1 < G) {
            o1[d] = E::bits(acc[mt][1] * il1);
            o1[d + 8] = E::bits(acc[mt][3] * il1);
          }
        }
      } else {
        const int slot = seg == 0 ? 0 : 1;
        const long long base = ((static_cast<long long>(gy) * p.N + c) * 2 + slot) * HG + w * G;
        float* o0 = p.part_o + (base + n0) * D;
        float* o1 = o0 + D;
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
          const int d = mt * 16 + g4;
          if (n0 < G) {
            o0[d] = acc[mt][0] * il0;
            o0[d + 8] = acc[mt][2] * il0;
          }
          if (n1 < G) {
            o1[d] = acc[mt][1] * il1;
            o1[d + 8] = acc[mt][3] * il1;
          }
        }
        if (g4 == 0) {
          if (n0 < G) p.part_lse[base + n0] = m0 + log2f(L0);
          if (n1 < G) p.part_lse[base + n1] = m1 + log2f(L1);
        }
        if constexpr (FUSED) {
          __syncwarp();
          if (lane == 0) mbar_arrive(pready);  // the merge warp counts it
          ++npart;
        }
      }
    }
  }
  if constexpr (FUSED) {
    // Rows whose last partial result this CTA delivered: merge all pieces.
    if (npart > 0) {
      if (!mbar_wait(mdone, 0)) {
        if (lane == 0) flag_error(p.err_flag, VH_ERR_TIMEOUT);
        return;
      }
      const int nv = *reinterpret_cast<volatile int*>(misc + kMiscNVerdict);
      uint32_t mphase = 0;
      for (int k = 0; k < nv; ++k) {
        const int* v = misc + kMiscVerdict + 5 * k;
        if (!v[0]) continue;
        const int np = v[3] - v[2] + 1;
        uint16_t* orow = p.out + (static_cast<long long>(v[1]) * p.Hq + static_cast<long long>(h) * G) * D;
        if (np > 32 / G) {
          // rows of many pieces (three or more batches of register loads): bring the
          // pieces in through the warp's free stage slices, 2 KB bulk copies
          if (!merge_pieces_staged<D, G, E>(p.part_lse, p.part_o, static_cast<long long>(gy) * p.N * 2, HG, w * G,
                                            v[2], np, v[4], orow, lane, smem_addr(smem), p.stage_bytes, S, Hc, w,
                                            smem_addr(bars + 2 * S + 5 + w), mphase)) {
            if (lane == 0) flag_error(p.err_flag, VH_ERR_TIMEOUT);
            return;
          }
        } else {
          merge_pieces<D, G, E>(p.part_lse, p.part_o, static_cast<long long>(gy) * p.N * 2, HG, w * G, v[2], np,
                             v[4], orow, lane);
        }
      }
    }
  }
}


// Per-step plan: the work list every attention launch of a decode step
// derives from the same lengths and page table, computed once.  CTA c of the
// grid (one per attention CTA) runs the attention kernel's own prologue
// arithmetic (tile counts, prefix sum, equal ranges) and writes its record:
// tile range, first and last row, and the page ids of the range's first
// kPlanWindow tiles; CTA 0 also writes the header and the per-row arrays.
// The kernel never releases its dependents early, and every thread ends with
// a GPU-scope fence after its last plan write, so by the time the last CTA
// has exited (when a programmatic dependent may start) the whole plan is
// visible: every kernel after it on the stream may read the plan before its
// own dependency wait.
__global__ void __launch_bounds__(256) decode_plan_kernel(const PlanParams p) {
  extern __shared__ int plan_smem[];  // warp totals [32], then cum [B + 1] (all shared memory is dynamic)
  int* warp_tot = plan_smem;
  int* pcum = plan_smem + 32;
  const int tid = threadIdx.x, c = blockIdx.x;
  const int max_len = p.max_pages_per_seq * p.P;
  int* g_len = p.rows + p.len_idx;
  int* g_pos = p.rows + p.pos_idx;
  for (int b = tid; b < p.B; b += blockDim.x) {
    const int a = p.active[b], L = p.seq_lens[b];
    int nt = row_tiles(a, L, max_len);
    if (a && nt == 0 && c == 0) flag_error(p.err_flag, VH_ERR_SEQLEN);
    int pos = 0;
    if (p.fused && nt > 0) {
      pos = p.positions ? p.positions[b] : L - 1;
      if (pos < 0 || pos >= p.max_pos) {
        nt = 0;
        if (c == 0) flag_error(p.err_flag, VH_ERR_POS);
      }
    }
    pcum[1 + b] = nt;
    if (c == 0) {
      g_len[b] = L;
      g_pos[b] = pos;
    }
  }
  if (tid == 0) pcum[0] = 0;
  __syncthreads();
  block_inclusive_scan(pcum, p.B, warp_tot);
  const long long T = pcum[p.B];
  const int n_eff = T == 0 ? 0 : min(p.N, (static_cast<int>(T) + p.min_tiles - 1) / p.min_tiles);
  int t0 = 0, t1 = 0, b0 = 0, bl = 0;
  // first row with cum[row + 1] > tt, among rows lo .. B-1
  auto row_of = [&](int lo, long long tt) -> int {
    int hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (pcum[mid + 1] > tt) hi = mid; else lo = mid + 1;
    }
    return lo;
  };
  if (c < n_eff) {
    t0 = static_cast<int>(range_begin(c, n_eff, T));
    t1 = static_cast<int>(range_begin(c + 1, n_eff, T));
    b0 = row_of(0, t0);
    bl = row_of(b0, t1 - 1);
  }
  int* rec = p.recs + static_cast<long long>(c) * kPlanRecInts;
  if (tid == 0) *reinterpret_cast<int4*>(rec) = make_int4(t0, t1, b0, bl);
  const bool p8 = (p.P == 8);
  const int tpp = (p.P + kTile - 1) / kTile;
  for (int i = tid; i < 2 * kPlanWindow; i += blockDim.x) {
    const int half = i / kPlanWindow;
    const long long tt = t0 + i % kPlanWindow;
    int pg = 0;
    if (tt < t1 && (half == 0 || p8)) {
      const int lo = row_of(b0, tt);
      pg = tile_page_id(p.page_table, p.max_pages_per_seq, p8, tpp, lo, static_cast<int>(tt - pcum[lo]), half);
    }
    rec[4 + i] = pg;
  }
  if (c == 0) {
    for (int b = tid; b <= p.B; b += blockDim.x) p.rows[b] = pcum[b];
    if (tid == 0) {
      reinterpret_cast<int4*>(p.hdr)[0] = make_int4(kPlanMagic, p.B, p.N, static_cast<int>(T));
      reinterpret_cast<int4*>(p.hdr)[1] = make_int4(n_eff, p.fused, p.max_pages_per_seq, p.P);
    }
  }
  // the plan's writes are performed at GPU scope before this thread exits
  // (a dependent's reads before its own wait are ordered only by this)
  __threadfence();
}

// Three-call path: one CTA per (row, kv-head group), one warp per kv head of
// the group (its G q heads).  Rows that one CTA finished, and padding rows,
// return at once.
template <int D, int G, typename E>
__global__ void __launch_bounds__(256) decode_combine_kernel(const CombineParams p) {
  pdl_wait();  // launched as a dependent of the attention kernel
  const int b = blockIdx.x, gy = blockIdx.y;
  const int4 pl = p.plan[b];
  if (pl.x < 0 || pl.x == pl.y) return;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int HG = p.Hc * G;
  merge_pieces<D, G, E>(p.part_lse, p.part_o, static_cast<long long>(gy) * p.N * 2, HG, w * G, pl.x, pl.y - pl.x + 1,
                     pl.z, p.out + (static_cast<long long>(b) * p.Hq + static_cast<long long>(gy) * HG + w * G) * D,
                     lane);
}

template <int D, int G, typename E>
const void* attn_kernel_ptr(bool fused) {
  return fused ? reinterpret_cast<const void*>(&decode_attn_kernel<D, G, true, E>)
               : reinterpret_cast<const void*>(&decode_attn_kernel<D, G, false, E>);
}

template <typename E>
const void* select_attn_kernel_t(int D, int G, bool fused) {
  if (D == 128) {
    switch (G) {
      case 1: return attn_kernel_ptr<128, 1, E>(fused);
      case 2: return attn_kernel_ptr<128, 2, E>(fused);
      case 4: return attn_kernel_ptr<128, 4, E>(fused);
      case 8: return attn_kernel_ptr<128, 8, E>(fused);
    }
  } else if (D == 64) {
    switch (G) {
      case 1: return attn_kernel_ptr<64, 1, E>(fused);
      case 2: return attn_kernel_ptr<64, 2, E>(fused);
      case 4: return attn_kernel_ptr<64, 4, E>(fused);
      case 8: return attn_kernel_ptr<64, 8, E>(fused);
    }
  }
  return nullptr;
}

const void* select_attn_kernel(int D, int G, bool fused, bool f16) {
  return f16 ? select_attn_kernel_t<ElemF16>(D, G, fused) : select_attn_kernel_t<ElemBf16>(D, G, fused);
}

}  // namespace

cudaError_t prepare_decode_attn(int D, int G, int max_smem) {
  for (bool f16 : {false, true})
    for (bool fused : {false, true}) {
      const void* k = select_attn_kernel(D, G, fused, f16);
      if (!k) return cudaErrorInvalidValue;
      const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

cudaError_t decode_attn_occupancy(const AttnParams& p, int* blocks_per_sm) {
  const void* k = select_attn_kernel(p.D, p.G, p.fused != 0, p.f16 != 0);
  if (!k) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, 32 * (p.Hc + (p.fused ? 2 : 1)),
                                                       p.smem_bytes);
}

cudaError_t launch_decode_attn(const AttnParams& p, cudaStream_t stream, bool pdl) {
  const void* k = select_attn_kernel(p.D, p.G, p.fused != 0, p.f16 != 0);
  if (!k) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.N, p.groups);
  cfg.blockDim = dim3(32 * (p.Hc + (p.fused ? 2 : 1)));
  cfg.dynamicSmemBytes = static_cast<size_t>(p.smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  void* args[] = {const_cast<AttnParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, k, args);
}

cudaError_t prepare_decode_plan(int max_smem) {
  return cudaFuncSetAttribute(decode_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

cudaError_t launch_decode_plan(const PlanParams& p, cudaStream_t stream) {
  // an ordinary launch (no programmatic dependency): it waits for all earlier
  // work on the stream
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.N);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 4 * (32 + static_cast<size_t>(p.B) + 1);
  cfg.stream = stream;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, decode_plan_kernel, p);
}

cudaError_t launch_decode_combine(const CombineParams& p, int groups, cudaStream_t stream) {
  // a programmatic dependent of the attention kernel that precedes it on the stream
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.B, groups);
  cfg.blockDim = dim3(32 * p.Hc);
  cfg.stream = stream;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
#define VH_COMBINE_CASE(DD, GG)                                                                             \
  if (p.D == DD && p.G == GG)                                                                               \
    return p.f16 ? cudaLaunchKernelEx(&cfg, decode_combine_kernel<DD, GG, ElemF16>, p)                      \
                 : cudaLaunchKernelEx(&cfg, decode_combine_kernel<DD, GG, ElemBf16>, p);
  VH_COMBINE_CASE(128, 1)
  VH_COMBINE_CASE(128, 2)
  VH_COMBINE_CASE(128, 4)
  VH_COMBINE_CASE(128, 8)
  VH_COMBINE_CASE(64, 1)
  VH_COMBINE_CASE(64, 2)
  VH_COMBINE_CASE(64, 4)
  VH_COMBINE_CASE(64, 8)
#undef VH_COMBINE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace vh
