// vh_common.cuh -- device helpers shared by the decode kernels (sm_103a).
//
// Inline PTX for the Blackwell data movers used here: mbarrier phase waits
// with a time limit, and the bulk (TMA, non-tensor) global->shared copy that
// completes on an mbarrier transaction count.  Plus bf16 / fp16 unpacking,
// rounding and tensor-core products, and the packed two-lane fp32 FMA of
// sm_100-class GPUs.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/vh.h"

namespace vh {

// A pipeline wait gives up after this many SM clock cycles (about 1 s at
// 2 GHz).  A wait that long only happens if something is broken; the kernel
// then records VH_ERR_TIMEOUT and winds down instead of hanging the GPU.
constexpr long long kWaitLimitCycles = 2000000000LL;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false if the
// time limit ran out first.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && clock64() - t0 > kWaitLimitCycles) return false;
  }
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to this CTA's shared memory; completion is signalled as a
// transaction count on mbarrier `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Tiled tensor copy of one 4-D box from global memory, described by a tensor
// map (in kernel-parameter space), into this CTA's shared memory; completion
// is signalled as a transaction count on mbarrier `bar`.  c0 is the innermost
// coordinate (in elements; c0 * element size must be a multiple of 16 bytes).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// The same copy with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const void* tmap, int c0, int c1, int c2, int c3,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
      "{%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policy for data read once: its lines are the first to be evicted.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Prefetch one box of a tiled tensor into L2 (no shared memory and no
// completion signal); a later copy of the same box is then served from L2.
__device__ __forceinline__ void tma_prefetch_l2_4d(const void* tmap, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(tmap), "r"(c0),
               "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a box stored with the
// 128-byte swizzle (rows of 128 bytes, box base 1024-byte aligned): the chunk
// index is XORed with the row index modulo 8, so the 8 rows an ldmatrix reads
// at the same logical chunk fall in 8 different bank groups.
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Two bf16 packed in a 32-bit word -> two exact fp32 values (low half first).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// d = a * b + c on two fp32 lanes at once (one instruction on sm_100-class GPUs),
// each lane rounded to nearest even like fmaf.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long ra, rb, rc, rd;
  ra = (static_cast<unsigned long long>(__float_as_uint(a.y)) << 32) | __float_as_uint(a.x);
  rb = (static_cast<unsigned long long>(__float_as_uint(b.y)) << 32) | __float_as_uint(b.x);
  rc = (static_cast<unsigned long long>(__float_as_uint(c.y)) << 32) | __float_as_uint(c.x);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  return make_float2(__uint_as_float(static_cast<uint32_t>(rd)),
                     __uint_as_float(static_cast<uint32_t>(rd >> 32)));
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  unsigned long long ra, rb, rd;
  ra = (static_cast<unsigned long long>(__float_as_uint(a.y)) << 32) | __float_as_uint(a.x);
  rb = (static_cast<unsigned long long>(__float_as_uint(b.y)) << 32) | __float_as_uint(b.x);
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  return make_float2(__uint_as_float(static_cast<uint32_t>(rd)),
                     __uint_as_float(static_cast<uint32_t>(rd >> 32)));
}

// fp32 -> bf16 bit pattern, round to nearest even (NaN stays NaN).
__device__ __forceinline__ uint32_t float_to_bf16_bits(float f) {
  unsigned short h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---- warp-level tensor-core helpers (sm_80+ forms, valid on sm_103a) -------

// Four 8x8 bf16 matrices from shared memory; lane l gives the address of row
// l % 8 of matrix l / 8, and receives row l / 4, columns 2 (l % 4) and
// 2 (l % 4) + 1 of each matrix.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Same, each 8x8 matrix transposed on the way in.
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Transpose one 8x8 bf16 matrix held in the ldmatrix fragment layout.
__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// c += a (16x16, row) * b (16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Split two fp32 values into bf16 high parts and bf16 residuals: x = hi + lo
// with |x - hi - lo| <= 2^-16 |x| (RNE at each step).
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(x0, x1);
  const float2 h = bf16x2_to_float2(hi);
  lo = pack_bf16x2(x0 - h.x, x1 - h.y);
}

// fp16 counterparts of the conversions above (IEEE binary16, round to nearest even).
__device__ __forceinline__ float2 f16x2_to_float2(uint32_t w) {
  float a, b;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(a), "=f"(b)
      : "r"(w));
  return make_float2(a, b);
}

__device__ __forceinline__ uint32_t float_to_f16_bits(float f) {
  unsigned short h;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// c += a (16x16, row) * b (16x8, col), fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Element type of q, k, v, the cache and the output: bf16 or fp16, both
// 16-bit patterns in memory.  The kernels are written once against this
// interface: unpacking, rounding (RNE), the hi + residual split of an fp32
// operand, and the tensor-core product of that type.
struct ElemBf16 {
  static constexpr bool kF16 = false;
  static __device__ __forceinline__ float2 to_float2(uint32_t w) { return bf16x2_to_float2(w); }
  static __device__ __forceinline__ float to_float(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }
  static __device__ __forceinline__ uint16_t bits(float f) { return static_cast<uint16_t>(float_to_bf16_bits(f)); }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) { return pack_bf16x2(lo, hi); }
  static __device__ __forceinline__ void mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    mma_bf16(c, a0, a1, a2, a3, b0, b1);
  }
};

struct ElemF16 {
  static constexpr bool kF16 = true;
  static __device__ __forceinline__ float2 to_float2(uint32_t w) { return f16x2_to_float2(w); }
  static __device__ __forceinline__ float to_float(uint16_t h) { return f16x2_to_float2(h).x; }
  static __device__ __forceinline__ uint16_t bits(float f) { return static_cast<uint16_t>(float_to_f16_bits(f)); }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) { return pack_f16x2(lo, hi); }
  static __device__ __forceinline__ void mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    mma_f16(c, a0, a1, a2, a3, b0, b1);
  }
};

// Split two fp32 values into a high part and a residual of element type E,
// x = hi + lo, both rounded to nearest even: bf16 keeps |x - hi - lo| <= 2^-16 |x|;
// fp16 keeps 2^-22 |x| for normal residuals, and an absolute 2^-25 once the
// residual is subnormal (the fp16 exponent range ends at 2^-14).
template <typename E>
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = E::pack2(x0, x1);
  const float2 h = E::to_float2(hi);
  lo = E::pack2(x0 - h.x, x1 - h.y);
}

// Programmatic dependent launch: let the next kernel on the stream start its
// CTAs early / wait until the previous kernel's results are visible.  Both are
// no-ops when the launches are not linked that way.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Barrier among `threads` threads (a multiple of 32) on hardware barrier `id`.
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// atomicAdd with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* addr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void flag_error(int32_t* err_flag, int bits) {
  if (err_flag != nullptr) atomicOr(err_flag, bits);
}

// Tiles are 16 consecutive tokens of one row; a page holds P/16 tiles.
constexpr int kTile = 16;

// Number of 16-token tiles a row contributes to the attention work list
// (0 for padding rows and for rows whose seq_len is out of range).
__device__ __forceinline__ int row_tiles(int active, int L, int max_len) {
  if (!active || L < 1 || L > max_len) return 0;
  return (L + kTile - 1) / kTile;
}

}  // namespace vh
