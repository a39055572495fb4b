// rope_append.cu -- RoPE table and the fused RoPE + KV-append kernel.
//
// Operation ("Adding a Model", vox-serve docs, section "1. The model code":
// keys and values are written into the paged cache before attention; RoPE is
// applied to q/k first; "Engineering TTS inference in vLLM-Omni", Qwen3-TTS
// section 4: RMSNorm variance and RoPE cos/sin in fp32): for each active row b
// at position pos = seq_len - 1 (or positions[b]),
//   q_rot[b]            = rope(norm_q(q[b]), pos)                 (fp32 out)
//   cache slot (L - 1)  = rne(rope(norm_k(k_new[b]), pos)), v_new[b]
// norm_*(x) = w * x / sqrt(mean(x^2) + eps) per head, in fp32, when weights
// are given (identity otherwise).  Rotation pair i (angle pos * theta^(-2i/D))
// is (i, i + D/2), or (2i, 2i + 1) with interleaved RoPE.  The 16-bit
// element type (bf16 or fp16; the Fish kernel takes either) is a template
// parameter; rne rounds to it.
//
// The work is tiny (a few hundred KB per call) and latency-bound: one CTA per
// row, 16-byte vector loads and stores, cos/sin read from a table built once
// in double precision so no per-call transcendental is evaluated.
#include "vh_common.cuh"
#include "vh_kernels.h"

namespace vh {

__global__ void rope_table_kernel(float* __restrict__ cos_sin, int max_pos, int D, double theta) {
  const int half = D / 2;
  const long long n = static_cast<long long>(max_pos) * half;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int p = static_cast<int>(idx / half);
    const int i = static_cast<int>(idx % half);
    const double f = pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(D));
    const double a = static_cast<double>(p) * f;
    double s, c;
    sincos(a, &s, &c);
    cos_sin[static_cast<long long>(p) * D + i] = static_cast<float>(c);
    cos_sin[static_cast<long long>(p) * D + half + i] = static_cast<float>(s);
  }
}

// One CTA per row (up to 1024 threads).  Work units: each thread rotates 4 consecutive pairs
// i..i+3 of one head (elements i..i+3 and i+D/2..i+D/2+3, or 2i..2i+7 interleaved);
// heads 0..Hq-1 are q heads (written to q_rot), heads Hq..Hq+Hkv-1 are the new k
// (written to the cache).  V is copied 16 bytes per thread.
template <typename E>
__global__ void __launch_bounds__(1024) rope_kv_append_kernel(RopeAppendParams p) {
  pdl_launch_dependents();  // an attention launch that depends on this one may start planning
  const int b = blockIdx.x;
  if (!p.active[b]) return;
  const int L = p.seq_lens[b];
  const int max_len = p.max_pages_per_seq * p.P;
  if (L < 1 || L > max_len) {
    if (threadIdx.x == 0) flag_error(p.err_flag, VH_ERR_SEQLEN);
    return;
  }
  const int pos = p.positions ? p.positions[b] : L - 1;
  if (pos < 0 || pos >= p.max_pos) {
    if (threadIdx.x == 0) flag_error(p.err_flag, VH_ERR_POS);
    return;
  }
  const int slot = L - 1;
  const long long lp = static_cast<long long>(b) * p.max_pages_per_seq + slot / p.P;
  const int page = p.page_table ? p.page_table[lp] : static_cast<int>(lp);  // no table: contiguous cache
  const bool page_ok = page >= 0 && page < p.num_pages;
  if (!page_ok && threadIdx.x == 0) flag_error(p.err_flag, VH_ERR_PAGE);
  const long long slot_off = static_cast<long long>(page) * p.page_stride +
                             static_cast<long long>(slot % p.P) * p.token_stride;

  const int D = p.D, half = D / 2;
  const int quads = half / 4;                  // 4-pair units per head (16 or 8: a head's units share a warp)
  const int heads = p.Hq + (page_ok ? p.Hkv : 0);
  const float* cs = p.cos_sin + static_cast<long long>(pos) * D;
  const int total = heads * quads;
  const bool ilv = p.rope_interleaved != 0;

  // every lane of a warp runs each round, so the per-head RMS reduction can shuffle
  for (int base = 0; base < total; base += blockDim.x) {
    const int u = base + threadIdx.x;
    const bool valid = u < total;
    const int h = valid ? u / quads : 0;
    const int i = valid ? (u % quads) * 4 : 0;
    const bool is_q = h < p.Hq;
    // x[k], y[k]: the two elements of pair i + k
    float x[4] = {0.f, 0.f, 0.f, 0.f}, y[4] = {0.f, 0.f, 0.f, 0.f};
    if (valid) {
      const uint16_t* src = is_q ? p.q + (static_cast<long long>(b) * p.Hq + h) * D
                                 : p.k_new + (static_cast<long long>(b) * p.Hkv + (h - p.Hq)) * D;
      if (ilv) {
        const uint4 w = *reinterpret_cast<const uint4*>(src + 2 * i);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 xy = E::to_float2(ws[k]);
          x[k] = xy.x;
          y[k] = xy.y;
        }
      } else {
        const uint2 lo = *reinterpret_cast<const uint2*>(src + i);
        const uint2 hi = *reinterpret_cast<const uint2*>(src + half + i);
        const float2 x01 = E::to_float2(lo.x), x23 = E::to_float2(lo.y);
        const float2 y01 = E::to_float2(hi.x), y23 = E::to_float2(hi.y);
        x[0] = x01.x; x[1] = x01.y; x[2] = x23.x; x[3] = x23.y;
        y[0] = y01.x; y[1] = y01.y; y[2] = y23.x; y[3] = y23.y;
      }
    }
    const float* nw = is_q ? p.q_norm_w : p.k_norm_w;
    // RMSNorm (fp32): the quads lanes of a head hold its D elements
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) ss += x[k] * x[k] + y[k] * y[k];
    for (int off = 1; off < quads; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (valid && nw != nullptr) {
      const float r = rsqrtf(ss / static_cast<float>(D) + p.norm_eps);
      float wx[4], wy[4];
      if (ilv) {
        const float4 wa = *reinterpret_cast<const float4*>(nw + 2 * i);
        const float4 wb = *reinterpret_cast<const float4*>(nw + 2 * i + 4);
        wx[0] = wa.x; wy[0] = wa.y; wx[1] = wa.z; wy[1] = wa.w;
        wx[2] = wb.x; wy[2] = wb.y; wx[3] = wb.z; wy[3] = wb.w;
      } else {
        const float4 wa = *reinterpret_cast<const float4*>(nw + i);
        const float4 wb = *reinterpret_cast<const float4*>(nw + half + i);
        wx[0] = wa.x; wx[1] = wa.y; wx[2] = wa.z; wx[3] = wa.w;
        wy[0] = wb.x; wy[1] = wb.y; wy[2] = wb.z; wy[3] = wb.w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[k] = wx[k] * (x[k] * r);
        y[k] = wy[k] * (y[k] * r);
      }
    }
    if (!valid) continue;
    const float4 c = *reinterpret_cast<const float4*>(cs + i);
    const float4 s = *reinterpret_cast<const float4*>(cs + half + i);
    const float cc[4] = {c.x, c.y, c.z, c.w};
    const float ss4[4] = {s.x, s.y, s.z, s.w};
    float rx[4], ry[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      rx[k] = x[k] * cc[k] - y[k] * ss4[k];
      ry[k] = y[k] * cc[k] + x[k] * ss4[k];
    }
    if (is_q) {
      float* dst = p.q_rot + (static_cast<long long>(b) * p.Hq + h) * D;
      if (ilv) {
        *reinterpret_cast<float4*>(dst + 2 * i) = make_float4(rx[0], ry[0], rx[1], ry[1]);
        *reinterpret_cast<float4*>(dst + 2 * i + 4) = make_float4(rx[2], ry[2], rx[3], ry[3]);
      } else {
        *reinterpret_cast<float4*>(dst + i) = make_float4(rx[0], rx[1], rx[2], rx[3]);
        *reinterpret_cast<float4*>(dst + half + i) = make_float4(ry[0], ry[1], ry[2], ry[3]);
      }
    } else {
      uint16_t* dst = p.k_cache + slot_off + static_cast<long long>(h - p.Hq) * p.head_stride;
      if (ilv) {
        *reinterpret_cast<uint4*>(dst + 2 * i) = make_uint4(E::pack2(rx[0], ry[0]), E::pack2(rx[1], ry[1]),
                                                            E::pack2(rx[2], ry[2]), E::pack2(rx[3], ry[3]));
      } else {
        *reinterpret_cast<uint2*>(dst + i) = make_uint2(E::pack2(rx[0], rx[1]), E::pack2(rx[2], rx[3]));
        *reinterpret_cast<uint2*>(dst + half + i) = make_uint2(E::pack2(ry[0], ry[1]), E::pack2(ry[2], ry[3]));
      }
    }
  }
  if (!page_ok) return;
  // V: Hkv*D 16-bit elements contiguous in v_new, head h at h*head_stride in
  // the slot; 8 per thread.
  const int nvec = p.Hkv * D / 8;
  const uint4* vsrc = reinterpret_cast<const uint4*>(p.v_new + static_cast<long long>(b) * p.Hkv * D);
  for (int u = threadIdx.x; u < nvec; u += blockDim.x) {
    const int h = (u * 8) / D, d = (u * 8) % D;
    *reinterpret_cast<uint4*>(p.v_cache + slot_off + static_cast<long long>(h) * p.head_stride + d) = vsrc[u];
  }
}

// The library's bounded pipeline wait on a barrier that nothing ever arrives
// on: it must give up after its time limit and report VH_ERR_TIMEOUT, leaving
// the context usable (the failure path of every pipeline wait).
__global__ void wait_timeout_selftest_kernel(int32_t* err_flag) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (!mbar_wait(smem_addr(&bar), 0) && threadIdx.x == 0) flag_error(err_flag, VH_ERR_TIMEOUT);
}

cudaError_t launch_wait_timeout_selftest(int32_t* err_flag, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(err_flag);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float* cos_sin, int max_pos, int D, double theta, cudaStream_t stream) {
  const long long n = static_cast<long long>(max_pos) * (D / 2);
  int blocks = static_cast<int>((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  rope_table_kernel<<<blocks, 256, 0, stream>>>(cos_sin, max_pos, D, theta);
  return cudaGetLastError();
}

cudaError_t launch_rope_kv_append(const RopeAppendParams& p, cudaStream_t stream) {
  // one pass over all heads of a row when it fits in one CTA (a thread per 4 rotation pairs)
  const int units = (p.Hq + p.Hkv) * (p.D / 8);
  int threads = ((units + 31) / 32) * 32;
  threads = threads < 128 ? 128 : (threads > 1024 ? 1024 : threads);
  if (p.f16)
    rope_kv_append_kernel<ElemF16><<<p.B, threads, 0, stream>>>(p);
  else
    rope_kv_append_kernel<ElemBf16><<<p.B, threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace vh
