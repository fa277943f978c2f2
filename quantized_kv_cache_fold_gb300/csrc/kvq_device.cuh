// Device helpers for the kvq kernels (sm_103a): inline PTX wrappers for mbarriers,
// bulk asynchronous copies, warp-level tensor-core MMA, ldmatrix/movmatrix, and the
// 4-bit / e4m3 -> fp16 register conversions.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "kvq.h"

namespace kvq {

constexpr int kD = 128;          // head dim
constexpr int kPage = 64;        // tokens per page
constexpr int kRec4 = 64;        // bytes per int4 token-head record
constexpr int kRec8 = 128;       // bytes per fp8 token-head record
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded waits give up after 2 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One arrival on `bar` from the threads with pred set (no branch around it).
__device__ __forceinline__ void mbar_arrive_if(uint64_t* bar, bool pred) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %1, 0;\n\t"
      "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_addr(bar)),
      "r"((uint32_t)pred)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may stay suspended (without issuing) for up to `hint_ns`
// while the phase is incomplete; it resumes as soon as the phase completes.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Non-blocking check of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed. Gives up after limit_ns
// (kWaitLimitNs unless a caller passes a shorter limit; 0: after the first unsuccessful
// try) or 2^30 polls and returns false; the caller records KVQ_DEVERR_TIMEOUT and abandons
// its work.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  if (limit_ns == 0) return false;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    // suspended while waiting (at most 20 us a try), so waiting warps take no issue slots
    if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
    if ((it & 15u) == 0 && globaltimer() - t0 > limit_ns) return false;
  }
  return false;
}

// ------------------------------------------------------------------ bulk copies

// One-dimensional bulk copy global -> shared through the TMA engine, completion counted
// on `bar` in bytes. Both addresses 16-byte aligned and bytes a multiple of 16 (page-head
// blocks of 4096/256/8192 bytes at 16-byte aligned bases, checked by the host).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// L2 policy for streamed KV pages: read once per decode step, so evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Named barrier among the first `nthreads` threads (consumer warps only).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ tensor cores (warp MMA)

// D += A(16x16, f16, row) * B(16x8, f16, col), fp32 accumulate.
// Fragments (g = lane/4, t = lane%4): a0 (row g, k 2t..2t+1), a1 (row g+8, k 2t..),
// a2 (row g, k 2t+8..), a3 (row g+8, k 2t+8..); b0 (k 2t..2t+1, n g), b1 (k 2t+8.., n g);
// d0,d1 (row g, n 2t, 2t+1), d2,d3 (row g+8, n 2t, 2t+1).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four 8x8 b16 matrices, transposed on load. Lane i gives the row address of row i%8 of
// matrix i/8; register k of thread (g = lane/4, t = lane%4) receives element [2t][g] in
// its low half and [2t+1][g] in its high half of matrix k.
// Four 8x8 b16 matrices in the mma fragment layout (lanes 8i..8i+7 give the row addresses of
// matrix i).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Transpose of an 8x8 b16 matrix held in the standard fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// ------------------------------------------------------------------ conversions

template <uint32_t LUT>
__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, %4;" : "=r"(d) : "r"(a), "r"(b), "r"(c), "n"(LUT));
  return d;
}

// Eight 4-bit codes n0..n7 (n_k in bits 4k..4k+3, one 32-bit word of a K record) -> four f16x2
// of exact f16 subnormals: h[0] = (n0, n4) 2^-24, h[1] = (n1, n5) 2^-20, h[2] = (n2, n6) 2^-24,
// h[3] = (n3, n7) 2^-20 (a nibble masked into an f16 with a zero exponent is its value times
// 2^-24; the high nibbles keep their place and so carry 16 n). Used for K against query fragments
// whose high-nibble slots are pre-divided by 16, so every product is q c 2^-24 exactly and the
// scores take one factor 2^24 with the per-token scale; no bias enters the fp32 sums.
__device__ __forceinline__ void unpack8_sub(uint32_t x, uint32_t (&h)[4]) {
  const uint32_t x8 = x >> 8;
  h[0] = x & 0x000F000Fu;
  h[1] = x & 0x00F000F0u;
  h[2] = x8 & 0x000F000Fu;
  h[3] = x8 & 0x00F000F0u;
}

// Physical position of the 16-byte chunk c (0..3) of the K record of token slot `slot`: chunk
// c ^ k_chunk_swz(slot). The XOR (bit 1 of the slot, and bit 3 of the slot as bit 1) spreads the
// shared-memory reads of the attention kernels over all 32 banks, both for a warp reading one
// chunk of 8 consecutive slots per quarter (split kernel) and for threads that each read whole
// records of the slots 16k + {0,1,8,9,2,3,10,11,...} (tcgen05 kernel).
__host__ __device__ __forceinline__ int k_chunk_swz(int slot) { return ((slot >> 1) & 1) | ((slot >> 2) & 2); }

// V code records: each 16-bit element holds the codes c0..c3 of dims 4j..4j+3 of one token in
// an encoding that converts to exact f16 without f16 arithmetic. Code c is taken as
// c - 7.5 = +-(e + 1/2), sign = (c < 8), e = c >= 8 ? c - 8 : 7 - c, and read as the f16
// subnormal +-(2e + 1) 2^(k - 24) = (c - 7.5) 2^(k - 23), for a per-dim k:
//   dim 4j+0: e in bits 1-3,   sign in bit 15   k = 0, read in place
//   dim 4j+1: e in bits 4-6,   sign in bit 14   k = 4, read after << 1
//   dim 4j+2: e in bits 11-13, sign in bit 7    k = 2, read after swapping the two bytes
//   dim 4j+3: e in bits 8-10,  sign in bit 0    k = 6, read after the swap and << 7
// The logical codes are what the cache stores; this is only their bit placement.
__host__ __device__ __forceinline__ uint32_t v_encode4(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3) {
  const uint32_t s0 = c0 < 8u, s1 = c1 < 8u, s2 = c2 < 8u, s3 = c3 < 8u;
  const uint32_t e0 = s0 ? 7u - c0 : c0 - 8u, e1 = s1 ? 7u - c1 : c1 - 8u;
  const uint32_t e2 = s2 ? 7u - c2 : c2 - 8u, e3 = s3 ? 7u - c3 : c3 - 8u;
  return (e0 << 1) | (s0 << 15) | (e1 << 4) | (s1 << 14) | (e2 << 11) | (s2 << 7) | (e3 << 8) | s3;
}
// Factor that takes dim 4j+i of a PV product over unpack8_v values back to c - 7.5 units: 2^(23 - k_i).
__device__ __forceinline__ float v_unscale(int i) {
  return i == 0 ? 8388608.0f : i == 1 ? 524288.0f : i == 2 ? 2097152.0f : 131072.0f;
}

// Two 16-bit V elements (two tokens, or dims 4j..4j+3 and 4j+4..4j+7 of one token) -> four f16x2:
// h[i] = dim 4j+i of the low element and of the high element, (c - 7.5) 2^(k_i - 23).
__device__ __forceinline__ void unpack8_v(uint32_t x, uint32_t (&h)[4]) {
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, 0x2301;" : "=r"(r) : "r"(x));  // bytes swapped within each half
  h[0] = lop3<0xEA>(x, 0x800E800Eu, 0x00010001u);
  h[1] = lop3<0xEA>(x << 1, 0x80E080E0u, 0x00100010u);
  h[2] = lop3<0xEA>(r, 0x80388038u, 0x00040004u);
  h[3] = lop3<0xEA>(r << 7, 0x83808380u, 0x00400040u);
}

// Two e4m3 bytes (low byte first) -> f16x2 (exact: e4m3 is a subset of f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t d;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(d) : "r"(two_bytes));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (lo, hi) fp32 -> f16x2, round to nearest even; lo in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// (lo, hi) fp32 -> f16x2, round to nearest even, saturating to +-65504 instead of overflowing.
__device__ __forceinline__ uint32_t pack_f16x2_sat(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// (lo, hi) fp32 -> two e4m3 bytes (lo in the low byte), nearest even, saturating finite.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ packed fp32 pairs
// Two fp32 values in one 64-bit register (lo in the low half). The .f32x2 forms of fma, add
// and mul round each half exactly as the scalar fma.rn / add.rn / mul.rn do, so a pair op gives
// the same bits as two scalar ops, in one instruction.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// Maximum of v over the 32 lanes of the warp (every lane active), in one instruction.
__device__ __forceinline__ float warp_max_all(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Sum / max over the 8 lanes that share (lane & 3): the lanes holding one accumulator
// column of an m16n8 MMA tile.
__device__ __forceinline__ float warp_sum_g(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

__device__ __forceinline__ float warp_max_g(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
  return v;
}

__device__ __forceinline__ void set_err(int32_t* dev_err, int bits) {
  if (dev_err) atomicOr(dev_err, bits);
}

// FP8 cache write (stock format): lane l's four elements of a 128-element row as e4m3(x /
// scale) -- IEEE division, nearest even, saturating -- packed low element first.
__device__ __forceinline__ uint32_t fp8_encode4(const float (&x)[4], float scale) {
  const uint32_t lo = pack_e4m3x2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale));
  const uint32_t hi = pack_e4m3x2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale));
  return lo | (hi << 16);
}

// Byte offset of lane l's four codes of the record in `slot` within a 64-slot ring block
// half (K or V): the record's 16-byte chunks are stored in XOR order (chunk c at c ^ (slot & 7)).
__device__ __forceinline__ int fp8_lane_offset(int slot, int lane) {
  return (slot % kPage) * kRec8 + ((lane >> 2) ^ (slot & 7)) * 16 + ((4 * lane) & 15);
}

__device__ __forceinline__ void fp8_store_row(uint8_t* block_half, int slot, const float (&x)[4], float scale,
                                              int lane) {
  *reinterpret_cast<uint32_t*>(block_half + fp8_lane_offset(slot, lane)) = fp8_encode4(x, scale);
}

// Lane l's four elements of row `row` of a [rows][128] tensor of fp32 or bf16.
__device__ __forceinline__ void load_row4(const void* base, int bf16, size_t row, int lane, float (&x)[4]) {
  if (bf16) {
    const uint2 u = reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + row * kD)[lane];
    x[0] = bf16_bits_to_f32(u.x & 0xFFFFu);
    x[1] = bf16_bits_to_f32(u.x >> 16);
    x[2] = bf16_bits_to_f32(u.y & 0xFFFFu);
    x[3] = bf16_bits_to_f32(u.y >> 16);
  } else {
    const float4 f = reinterpret_cast<const float4*>(static_cast<const float*>(base) + row * kD)[lane];
    x[0] = f.x;
    x[1] = f.y;
    x[2] = f.z;
    x[3] = f.w;
  }
}

__device__ __forceinline__ bool warp_all_finite(const float (&x)[4]) {
  const bool ok = isfinite(x[0]) && isfinite(x[1]) && isfinite(x[2]) && isfinite(x[3]);
  return __all_sync(0xffffffffu, ok);
}

// Orders this thread's generic-proxy global writes before later async-proxy (bulk copy) reads.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later async-proxy ones
// (a bulk copy refilling a stage that was patched with ordinary stores).
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ thread-block clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_cluster(uint32_t shared_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(shared_addr), "r"(rank));
  return r;
}

// Split cluster barrier: arrive early (relaxed), wait later (acquire). Here it publishes
// mbarrier initialisation (after fence_barrier_init) to the other CTAs of the cluster.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Asynchronous stores into another CTA's shared memory (cluster addresses from map_cluster);
// each completes its byte count on that CTA's mbarrier `bar`.
__device__ __forceinline__ void st_async_f32x2(uint32_t addr, float a, float b, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "f"(a), "f"(b), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void st_async_f32x4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
               : "memory");
}

// Pull one 128-byte line into L1 ahead of its use.
__device__ __forceinline__ void prefetch_l1(const void* p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }

// Warm L2 with `bytes` (a multiple of 16) at a 16-byte aligned global address. Nothing is
// read into the SM, so this is safe while another grid may still be writing the data.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// ------------------------------------------------------------------ tcgen05 (tensor memory)

// Shared-memory descriptor of a tcgen05.mma operand in the 128-byte-swizzle layout: rows of 128
// bytes in 8-row atoms on 1024-byte boundaries, 16-byte chunk c of row r stored at chunk
// c ^ (r & 7). K-major operands: sbo = stride between 8-row groups, lbo unused, the next 16
// elements of K start 32 bytes further. MN-major operands: lbo = stride between 64-element MN
// atoms, sbo = stride between 8-row K groups.
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma.kind::f16: f16 A and B, f32 accumulator, M = 128, N
// (multiple of 16, <= 256); a_mn / b_mn select MN-major operands.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int n, bool a_mn, bool b_mn) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
         ((128u >> 4) << 24);
}

// D (tensor memory) = A B (+ D if accumulate), issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One arrival on `bar` once every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// D (tensor memory) = A B (+ D), with A read from tensor memory: row i of A in lane i, its K
// elements two per 32-bit column (element 2c in the low half of column c). Issued by one thread.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Registers per thread of the executing warpgroup (all four of its warps execute the same one).
template <int N>
__device__ __forceinline__ void reg_alloc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void reg_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// All 512 tensor-memory columns of the SM for this CTA (whole warp); the address lands in *dst.
__device__ __forceinline__ void tmem_alloc_512(uint32_t* dst) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_addr(dst)) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_512(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(taddr) : "memory");
}

// 16 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}
// 16 consecutive 32-bit columns of this thread's lane from raw words.
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// Four 16-lane x 8-column blocks (lanes taddr.lane .. +15, columns taddr.col + 8j ..): thread
// (g = lane/4, t = lane%4) gives r[4j] at (lane g, column 8j + 2t), r[4j+1] at (g, 8j + 2t + 1),
// r[4j+2] at (g + 8, 8j + 2t), r[4j+3] at (g + 8, 8j + 2t + 1) -- the mma.sync accumulator layout.
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Tensor-memory columns for the CTA (whole warp); the address lands in *dst.
__device__ __forceinline__ void tmem_alloc_256(uint32_t* dst) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_addr(dst)) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_256(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(taddr) : "memory");
}

// 4 consecutive 32-bit columns of this thread's lane (warp w reads lanes 32 (w % 4) + laneid).
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const float (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(__float_as_uint(v[0])),
               "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3]))
               : "memory");
}

// 8 consecutive 32-bit columns of this thread's lane (warp w reads lanes 32 (w % 4) + laneid).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Named barrier that also returns whether `pred` held in any / every participating thread.
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %3, 0;\n\t"
      "bar.red.or.pred q, %1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(nthreads), "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------ programmatic dependent launch

// Lets the next grid on the stream (launched with programmatic stream serialisation) start
// its prologue while this one runs.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until the preceding grid has completed and its memory operations are visible; a
// no-op when the grid was launched without programmatic serialisation.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace kvq
