// decode_attn.cu -- paged GQA decode attention (q_len = 1) and the LSE combine.
//
// Operation ("Engineering TTS inference in vLLM-Omni", Fish Speech S2 Pro,
// "model-specific attention kernel"): for every active row b and q head g,
// with kv head h = g / G,
//     s_j = scale * <q_rot[b,g], K[b,h,j]>,  j < L_b  (keys through the page table)
//     o   = sum_j softmax(s)_j V[b,h,j]
// in fp32 with a running max (online softmax); long rows are cut into
// segments whose partial (o, lse) are merged by the log-sum-exp recurrence.
//
// Design for GB300 (HBM-bound: 2-4 flops per byte of K/V):
//  * Work list.  Every active row contributes ceil(L/16) tiles of 16 tokens;
//    the list of all tiles in row order is cut into N equal contiguous
//    ranges, one per CTA, on the device (each CTA prefix-sums the row tile
//    counts in shared memory).  No host sync, static grid, and the load is
//    balanced to within one tile whatever the length mix; a row is split
//    where its tiles straddle two CTAs (at most two partial segments per CTA).
//  * Data movement.  One producer warp streams each tile into a ring of
//    shared-memory stages with bulk asynchronous copies (one 16-byte-aligned
//    copy per token row, K rows and V rows of the CTA's kv heads), completed
//    on an mbarrier transaction count; consumers release a stage through a
//    second mbarrier.  K rows get a 32-byte pad so the per-key reads of the
//    score step are free of bank conflicts.
//  * Compute.  One consumer warp per kv head.  Scores: a lane owns one key
//    (and half of D), q is read from shared memory as a broadcast, bf16 K is
//    widened with shifts and multiplied with packed two-lane fp32 FMAs.  The
//    value step: a lane owns 8 output dims for a subset of the tile's keys.
//    exp2 with log2(e) folded into the scale.
//  * Stale slots (tail of the last page, slots never copied) are never used:
//    their scores are replaced by -inf before the max and their V rows are
//    skipped, so NaN or Inf bits there cannot reach the output.
#include "vh_common.cuh"
#include "vh_kernels.h"

namespace vh {

namespace {

constexpr int kMaxHc = 8;                    // kv heads (consumer warps) per CTA
constexpr int kThreadsMax = 32 * (kMaxHc + 1);

template <int D, int G>
struct Lay {
  static constexpr int KSPLIT = 256 / D;          // key groups in the value step
  static constexpr int KPER = kTile / KSPLIT;     // keys per group
  static constexpr int CHUNKS = D / 8;            // 16-byte chunks of a head row
  static constexpr int PSTRIDE = kTile * G + KSPLIT * 4;  // floats of p per warp
  __device__ static __forceinline__ int pidx(int k) { return k * G + (k / KPER) * 4; }
};

__device__ __forceinline__ long long range_begin(int c, int n_eff, long long T) {
  return (static_cast<long long>(c) * T) / n_eff;
}

// CTA whose range [c T / n, (c+1) T / n) holds tile s.
__device__ __forceinline__ int cta_of(long long s, int n_eff, long long T) {
  return static_cast<int>(((s + 1) * n_eff - 1) / T);
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

enum { kMiscWarpTot = 0, kMiscAbort = 32, kMiscInts = 40 };

template <int D, int G>
__global__ void __launch_bounds__(kThreadsMax, 1) decode_attn_kernel(const AttnParams p) {
  using L_ = Lay<D, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hc = p.Hc, S = p.stages;
  const int c = blockIdx.x, gy = blockIdx.y;
  int* cum = reinterpret_cast<int*>(smem + p.cum_off);
  int* lens = reinterpret_cast<int*>(smem + p.len_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  int* misc = reinterpret_cast<int*>(smem + p.bar_off + 16 * S);
  volatile int* abort_flag = misc + kMiscAbort;
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + S);
  const int max_len = p.max_pages_per_seq * p.P;

  // ---- prologue: tile count of every row and their prefix sum -------------
  for (int b = tid; b < p.B; b += blockDim.x) {
    const int a = p.active[b], L = p.seq_lens[b];
    const int nt = row_tiles(a, L, max_len);
    cum[1 + b] = nt;
    lens[b] = L;
    if (a && nt == 0 && c == 0 && gy == 0) flag_error(p.err_flag, VH_ERR_SEQLEN);
  }
  if (tid == 0) {
    cum[0] = 0;
    *abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, Hc);
    }
    fence_barrier_init();
  }
  __syncthreads();
  block_inclusive_scan(cum, p.B, misc + kMiscWarpTot);
  const long long T = cum[p.B];
  const int n_eff = T == 0 ? 0 : static_cast<int>(min(static_cast<long long>(p.N), (T + p.min_tiles - 1) / p.min_tiles));

  // ---- per-row duties, rows b = c (mod N): split plan, zero padding rows ---
  const int HG = Hc * G;  // q heads of this CTA
  for (int b = c; b < p.B; b += p.N) {
    const int nt = cum[b + 1] - cum[b];
    if (nt == 0) {
      uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<long long>(b) * p.Hq + gy * HG) * D);
      for (int i = tid; i < HG * D / 8; i += blockDim.x) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      if (gy == 0 && tid == 0) p.plan[b] = make_int4(-1, -1, 0, 0);
    } else if (gy == 0 && tid == 0) {
      const long long s0 = cum[b], s1 = cum[b + 1] - 1;
      const int cf = cta_of(s0, n_eff, T), cl = cta_of(s1, n_eff, T);
      p.plan[b] = make_int4(cf, cl, range_begin(cf, n_eff, T) == s0 ? 0 : 1, nt);
    }
  }
  if (c >= n_eff) return;

  const long long t0 = range_begin(c, n_eff, T), t1 = range_begin(c + 1, n_eff, T);
  int b0;
  {
    int lo = 0, hi = p.B - 1;  // first row with cum[b + 1] > t0
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (cum[mid + 1] > t0) hi = mid; else lo = mid + 1;
    }
    b0 = lo;
  }
  unsigned char* stage_base = smem;

  if (warp == Hc) {
    // ======================= producer warp =================================
    const int h0 = gy * Hc;
    const unsigned char* kbase = reinterpret_cast<const unsigned char*>(p.k_cache + static_cast<long long>(h0) * D);
    const unsigned char* vbase = reinterpret_cast<const unsigned char*>(p.v_cache + static_cast<long long>(h0) * D);
    int b = b0;
    long long rt0 = cum[b], rt1 = cum[b + 1];
    int stage = 0, round = 0;
    long long issued = 0;
    bool aborted = false;
    for (long long t = t0; t < t1; ++t, ++issued) {
      while (t >= rt1) {
        ++b;
        rt0 = rt1;
        rt1 = cum[b + 1];
      }
      const int tok0 = static_cast<int>(t - rt0) * kTile;
      const int nvalid = min(kTile, lens[b] - tok0);
      int page = p.page_table[static_cast<long long>(b) * p.max_pages_per_seq + tok0 / p.P];
      if (page < 0 || page >= p.num_pages) {
        if (lane == 0) flag_error(p.err_flag, VH_ERR_PAGE);
        page = 0;
      }
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
      const uint32_t fb = full0 + 8 * stage;
      if (lane == 0) mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nvalid) * 2u * p.row_copy_bytes);
      __syncwarp();
      const int r = lane & 15;
      if (r < nvalid) {
        const long long off = 2LL * (static_cast<long long>(page) * p.page_stride +
                                     static_cast<long long>(tok0 % p.P + r) * p.token_stride);
        unsigned char* st = stage_base + static_cast<long long>(stage) * p.stage_bytes;
        if (lane < 16)
          bulk_g2s(smem_addr(st + r * p.k_row_bytes), kbase + off, p.row_copy_bytes, fb);
        else
          bulk_g2s(smem_addr(st + kTile * p.k_row_bytes + r * p.v_row_bytes), vbase + off, p.row_copy_bytes, fb);
      }
      if (++stage == S) {
        stage = 0;
        ++round;
      }
    }
    if (aborted) {
      // Let the copies already issued land before the CTA's shared memory goes away.
      const long long n = min(issued, static_cast<long long>(S));
      for (long long k = issued - n; k < issued; ++k)
        (void)mbar_wait(full0 + 8 * static_cast<int>(k % S), static_cast<uint32_t>((k / S) & 1));
    }
    return;
  }

  // ========================= consumer warps ==================================
  const int w = warp;                 // kv head within the CTA
  const int h = gy * Hc + w;          // kv head
  float* qs = reinterpret_cast<float*>(smem + p.q_off) + w * G * D;
  float* ps = reinterpret_cast<float*>(smem + p.p_off) + w * L_::PSTRIDE;
  const int kt = lane >> 1, khalf = lane & 1;        // score step: key, half of D
  const int chunk = lane % L_::CHUNKS, kp = lane / L_::CHUNKS;  // value step
  const float NEG_INF = __int_as_float(0xff800000);

  float m[G], lsum[G];
  float2 acc[G][4];
  int b = b0;
  long long rt0 = cum[b], rt1 = cum[b + 1];
  int seg = 0, stage = 0, round = 0;
  for (long long t = t0; t < t1; ++t) {
    bool new_row = false;
    while (t >= rt1) {
      ++b;
      rt0 = rt1;
      rt1 = cum[b + 1];
      new_row = true;
    }
    if (new_row) ++seg;
    const long long sb = max(t0, rt0), se = min(t1, rt1);
    if (t == sb) {
      const float* qsrc = p.q_rot + (static_cast<long long>(b) * p.Hq + static_cast<long long>(h) * G) * D;
      __syncwarp();
      for (int i = lane * 4; i < G * D; i += 128)
        *reinterpret_cast<float4*>(qs + i) = __ldg(reinterpret_cast<const float4*>(qsrc + i));
      __syncwarp();
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[g] = NEG_INF;
        lsum[g] = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[g][q] = make_float2(0.f, 0.f);
      }
    }
    const int tok0 = static_cast<int>(t - rt0) * kTile;
    const int nvalid = min(kTile, lens[b] - tok0);
    if (!mbar_wait(full0 + 8 * stage, round & 1)) {
      if (lane == 0) flag_error(p.err_flag, VH_ERR_TIMEOUT);
      *abort_flag = 1;
      return;
    }
    const unsigned char* st = stage_base + static_cast<long long>(stage) * p.stage_bytes;

    // ---- scores: lane (kt, khalf) dots its key with all G q heads --------------
    float s[G];
    {
      const unsigned char* krow = st + kt * p.k_row_bytes + w * D * 2;
      float2 a0[G], a1[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        a0[g] = make_float2(0.f, 0.f);
        a1[g] = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        const int cc = 2 * j + khalf;
        const uint4 kv = *reinterpret_cast<const uint4*>(krow + cc * 16);
        const float2 k0 = bf16x2_to_float2(kv.x), k1 = bf16x2_to_float2(kv.y);
        const float2 k2 = bf16x2_to_float2(kv.z), k3 = bf16x2_to_float2(kv.w);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qa = *reinterpret_cast<const float4*>(qs + g * D + cc * 8);
          const float4 qb = *reinterpret_cast<const float4*>(qs + g * D + cc * 8 + 4);
          a0[g] = ffma2(k0, make_float2(qa.x, qa.y), a0[g]);
          a1[g] = ffma2(k1, make_float2(qa.z, qa.w), a1[g]);
          a0[g] = ffma2(k2, make_float2(qb.x, qb.y), a0[g]);
          a1[g] = ffma2(k3, make_float2(qb.z, qb.w), a1[g]);
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float v = (a0[g].x + a0[g].y) + (a1[g].x + a1[g].y);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        s[g] = kt < nvalid ? v * p.scale_log2 : NEG_INF;
      }
    }

    // ---- online softmax update ----------------------------------------------
    float alpha[G];
    bool rescale = false;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mx = s[g];
#pragma unroll
      for (int off = 2; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[g], mx);
      alpha[g] = exp2f(m[g] - mn);
      rescale |= (alpha[g] != 1.f);
      s[g] = exp2f(s[g] - mn);  // p
      lsum[g] = lsum[g] * alpha[g] + s[g];
      m[g] = mn;
    }
    if (khalf == 0) {
      float* dst = ps + L_::pidx(kt);
      if constexpr (G == 1) {
        dst[0] = s[0];
      } else if constexpr (G == 2) {
        *reinterpret_cast<float2*>(dst) = make_float2(s[0], s[1]);
      } else {
#pragma unroll
        for (int g = 0; g < G; g += 4)
          *reinterpret_cast<float4*>(dst + g) = make_float4(s[g], s[g + 1], s[g + 2], s[g + 3]);
      }
    }
    __syncwarp();

    // ---- values: lane (chunk, kp) accumulates 8 dims over its keys -------------
    if (rescale) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float2 a2 = make_float2(alpha[g], alpha[g]);
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[g][q] = fmul2(acc[g][q], a2);
      }
    }
    {
      const unsigned char* vcol = st + kTile * p.k_row_bytes + w * D * 2 + chunk * 16;
#pragma unroll
      for (int i = 0; i < L_::KPER; ++i) {
        const int k = kp * L_::KPER + i;
        if (k < nvalid) {
          const uint4 vv = *reinterpret_cast<const uint4*>(vcol + k * p.v_row_bytes);
          const float2 v0 = bf16x2_to_float2(vv.x), v1 = bf16x2_to_float2(vv.y);
          const float2 v2 = bf16x2_to_float2(vv.z), v3 = bf16x2_to_float2(vv.w);
          float pg[G];
          const float* src = ps + L_::pidx(k);
          if constexpr (G == 1) {
            pg[0] = src[0];
          } else if constexpr (G == 2) {
            const float2 t2 = *reinterpret_cast<const float2*>(src);
            pg[0] = t2.x;
            pg[1] = t2.y;
          } else {
#pragma unroll
            for (int g = 0; g < G; g += 4) {
              const float4 t4 = *reinterpret_cast<const float4*>(src + g);
              pg[g] = t4.x;
              pg[g + 1] = t4.y;
              pg[g + 2] = t4.z;
              pg[g + 3] = t4.w;
            }
          }
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float2 pp = make_float2(pg[g], pg[g]);
            acc[g][0] = ffma2(v0, pp, acc[g][0]);
            acc[g][1] = ffma2(v1, pp, acc[g][1]);
            acc[g][2] = ffma2(v2, pp, acc[g][2]);
            acc[g][3] = ffma2(v3, pp, acc[g][3]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * stage);
    if (++stage == S) {
      stage = 0;
      ++round;
    }

    // ---- end of a segment: finished row or partial result ----------------------
    if (t == se - 1) {
#pragma unroll
      for (int off = L_::CHUNKS; off < 32; off <<= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[g][q].x += __shfl_xor_sync(0xffffffffu, acc[g][q].x, off);
            acc[g][q].y += __shfl_xor_sync(0xffffffffu, acc[g][q].y, off);
          }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int off = 2; off < 32; off <<= 1) lsum[g] += __shfl_xor_sync(0xffffffffu, lsum[g], off);
      }
      const bool full_row = (sb == rt0) && (se == rt1);
      if (full_row) {
        if (kp == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float il = 1.f / lsum[g];
            uint4 o;
            o.x = pack_bf16x2(acc[g][0].x * il, acc[g][0].y * il);
            o.y = pack_bf16x2(acc[g][1].x * il, acc[g][1].y * il);
            o.z = pack_bf16x2(acc[g][2].x * il, acc[g][2].y * il);
            o.w = pack_bf16x2(acc[g][3].x * il, acc[g][3].y * il);
            *reinterpret_cast<uint4*>(p.out + (static_cast<long long>(b) * p.Hq + h * G + g) * D + chunk * 8) = o;
          }
        }
      } else {
        const int slot = seg == 0 ? 0 : 1;
        const long long base = ((static_cast<long long>(gy) * p.N + c) * 2 + slot) * HG + w * G;
        if (kp == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float il = 1.f / lsum[g];
            float* dst = p.part_o + (base + g) * D + chunk * 8;
            *reinterpret_cast<float4*>(dst) =
                make_float4(acc[g][0].x * il, acc[g][0].y * il, acc[g][1].x * il, acc[g][1].y * il);
            *reinterpret_cast<float4*>(dst + 4) =
                make_float4(acc[g][2].x * il, acc[g][2].y * il, acc[g][3].x * il, acc[g][3].y * il);
          }
        }
        if (lane == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) p.part_lse[base + g] = m[g] + log2f(lsum[g]);
        }
      }
    }
  }
}

// One CTA per (row, kv-head group); a warp per q head.  Rows that one CTA
// finished (or padding rows) return at once.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const CombineParams p) {
  const int b = blockIdx.x, gy = blockIdx.y;
  const int4 pl = p.plan[b];
  if (pl.x < 0 || pl.x == pl.y) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int HG = p.Hc * p.G;
  constexpr int PER = D / 32;
  for (int lq = warp; lq < HG; lq += nw) {
    float M = __int_as_float(0xff800000);
    for (int cc = pl.x; cc <= pl.y; ++cc) {
      const int slot = cc == pl.x ? pl.z : 0;
      const long long idx = ((static_cast<long long>(gy) * p.N + cc) * 2 + slot) * HG + lq;
      M = fmaxf(M, p.part_lse[idx]);
    }
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    float wsum = 0.f;
    for (int cc = pl.x; cc <= pl.y; ++cc) {
      const int slot = cc == pl.x ? pl.z : 0;
      const long long idx = ((static_cast<long long>(gy) * p.N + cc) * 2 + slot) * HG + lq;
      const float wgt = exp2f(p.part_lse[idx] - M);
      wsum += wgt;
      const float* o = p.part_o + idx * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = *reinterpret_cast<const float4*>(o);
        acc[0] += wgt * v.x;
        acc[1] += wgt * v.y;
        acc[2] += wgt * v.z;
        acc[3] += wgt * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(o);
        acc[0] += wgt * v.x;
        acc[1] += wgt * v.y;
      }
    }
    const float iw = 1.f / wsum;
    uint16_t* dst = p.out + (static_cast<long long>(b) * p.Hq + gy * HG + lq) * D + lane * PER;
    if constexpr (PER == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[0] * iw, acc[1] * iw), pack_bf16x2(acc[2] * iw, acc[3] * iw));
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * iw, acc[1] * iw);
    }
  }
}

template <int D, int G>
const void* attn_kernel_ptr() {
  return reinterpret_cast<const void*>(&decode_attn_kernel<D, G>);
}

const void* select_attn_kernel(int D, int G) {
  if (D == 128) {
    switch (G) {
      case 1: return attn_kernel_ptr<128, 1>();
      case 2: return attn_kernel_ptr<128, 2>();
      case 4: return attn_kernel_ptr<128, 4>();
      case 8: return attn_kernel_ptr<128, 8>();
    }
  } else if (D == 64) {
    switch (G) {
      case 1: return attn_kernel_ptr<64, 1>();
      case 2: return attn_kernel_ptr<64, 2>();
      case 4: return attn_kernel_ptr<64, 4>();
      case 8: return attn_kernel_ptr<64, 8>();
    }
  }
  return nullptr;
}

}  // namespace

cudaError_t prepare_decode_attn(int D, int G, int max_smem) {
  const void* k = select_attn_kernel(D, G);
  if (!k) return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

cudaError_t decode_attn_occupancy(const AttnParams& p, int* blocks_per_sm) {
  const void* k = select_attn_kernel(p.D, p.G);
  if (!k) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, 32 * (p.Hc + 1), p.smem_bytes);
}

cudaError_t launch_decode_attn(const AttnParams& p, cudaStream_t stream) {
  const void* k = select_attn_kernel(p.D, p.G);
  if (!k) return cudaErrorInvalidValue;
  dim3 grid(p.N, p.groups), block(32 * (p.Hc + 1));
  void* args[] = {const_cast<AttnParams*>(&p)};
  return cudaLaunchKernel(k, grid, block, args, static_cast<size_t>(p.smem_bytes), stream);
}

cudaError_t launch_decode_combine(const CombineParams& p, int groups, cudaStream_t stream) {
  dim3 grid(p.B, groups);
  const int HG = p.Hc * p.G;
  const int threads = 32 * (HG < 8 ? HG : 8);
  if (p.D == 128)
    decode_combine_kernel<128><<<grid, threads, 0, stream>>>(p);
  else
    decode_combine_kernel<64><<<grid, threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace vh
