// FP8 sliding-window decode attention: one thread-block cluster per (sequence, KV head).
//
// "Serving Kolibri-1 with a 4-bit KV cache", section on the sliding-window layers: those
// layers keep the stock FP8 (e4m3) cache and attend over the newest `window` positions. The
// cache is a ring of `cap` slots per (sequence, KV head), position p in slot p mod cap, stored
// as 64-slot blocks of 16384 bytes (64 K records of 128 e4m3 codes, then 64 V records; the
// 16-byte chunks of slot s's record in XOR order, chunk c at c ^ (s & 7)).
//
// A window is a few hundred positions: far too little work to spread over a whole grid and
// merge through global memory, and far too much latency for one SM to pull and process alone.
// Here the ring is cut into 32-slot units spread over the warps of one cluster (at most 8
// CTAs), and the partial softmax states are merged on chip. With many (sequence, KV head)
// pairs (at least one per SM) the pairs themselves fill the GPU: then each pair gets one CTA
// (a cluster of one) whose few unit streams take several units each in turn (as many streams
// as keep the grid in its fewest waves of resident CTAs), and there is nothing to push:
//
//   warp (unit stream w, tile group tg): streams the units u = w, w + NS, w + 2 NS, ...
//     (NS = streams in the cluster) through its own one- or two-stage shared-memory buffer,
//     each unit two bulk copies (TMA engine; its 32 K records and its 32 V records)
//     completing on the warp's own mbarrier;
//     if the call appends rows, the stream owning a new row's unit encodes it (e4m3 of
//     x / scale), stores it into the ring for later steps (tile group 0 only) and patches
//     it into the landed copy, so the appended rows are attended in the same launch;
//     QK^T and PV on tensor cores (mma.m16n8k16, e4m3 -> f16 exactly), online softmax in
//     exp2 form, query rows masked outside [max(0, p_r - window + 1), p_r];
//   a lone stream in a cluster of one normalises its rows and stores them; otherwise
//   partial (m, l, acc[128]) per stream and query row -> shared memory;
//   each CTA merges its streams per (row, 8 dims) with log-sum-exp weights and pushes the
//   result into CTA 0 of the cluster with asynchronous remote stores (st.async) that complete
//   a byte count on CTA 0's receive mbarrier, then exits; CTA 0 waits for all bytes, merges
//   the cluster's partials from its own shared memory and writes the normalised output.
//
// Launch with programmatic stream serialisation: the prologue (barrier set-up and L2
// prefetches, which read nothing into the SM) may overlap the previous grid; everything else
// follows griddepcontrol.wait. Every mbarrier wait is bounded (KVQ_DEVERR_TIMEOUT). The one
// cluster barrier (arrive at start, wait before the first remote store) only publishes CTA
// 0's receive barrier, and every thread reaches both halves unconditionally.

#include <algorithm>
#include <cmath>

#include <mutex>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

// Unit streams (warps per query-tile group) per CTA.
#ifndef KVQ_SWA_STREAMS
#define KVQ_SWA_STREAMS 6
#endif
// Stages per unit stream in the one-CTA-per-pair plan.
#ifndef KVQ_SWA_BATCH_STAGES
#define KVQ_SWA_BATCH_STAGES 2
#endif
static_assert(KVQ_SWA_BATCH_STAGES >= 1 && KVQ_SWA_BATCH_STAGES <= 2, "a unit stream tracks at most two stages");

constexpr int kBlk = 2 * kPage * kRec8;  // 16384 bytes per 64-slot ring block (K half, V half)
constexpr int kUnit = 32;                // slots per work unit
constexpr int kHalf = kUnit * kRec8;     // 4096 bytes: one unit's K (or V) records
constexpr int kStg = 2 * kHalf;          // 8192 bytes per stage: the unit's K then V records
constexpr int kRedStride = 132;          // floats per partial row: m, l, 2 pad, acc[128] (16-byte aligned)
constexpr int kPushBytes = 8 + 4 * kD;   // bytes pushed per query row: (m, l) and acc
constexpr int kMaxCluster = 8;
constexpr int kMaxStreams = 8;           // unit streams per CTA (merge loops are unrolled to this)
constexpr int kMaxUnitsPerStream = 4;    // beyond this the split-K path with a combine pass is used
constexpr int kMaxUnitsBatched = 18;     // one-CTA-per-pair plan: a 576-slot ring through one stream
constexpr size_t kSmemCap = 200 * 1024;
constexpr float kLog2e = 1.4426950408889634f;

struct SwaParams {
  const uint8_t* ring;  // [num_seqs][Hkv][nblk][kBlk]
  int cap, nblk, nunits, window;
  int B, S, Hq, Hkv, G, R;
  const int32_t* pos0;
  const void* q;
  int bf16;  // q, k_new, v_new are bf16 (else fp32)
  const void* k_new;
  const void* v_new;
  float k_scale, v_scale, score_scale;
  float* out;
  int32_t* dev_err;
  int cs, nws, ntg, nst, rows_pad;
};

struct SwaPlan {
  int NT, ntg, nws, cs, nst, rows_pad, ups;
  bool batched;  // one CTA per pair, streams of up to kMaxUnitsBatched units
  size_t smem;
};

// Shared memory: stages [warp][nst][kStg], the warps' copy barriers [warp][nst] and the
// receive barrier, partials [warp][NT*8][132], the receive area [cs - 1][rows_pad][132] (CTA 0
// of the cluster receives from ranks 1 .. cs - 1).
struct SwaSmem {
  size_t bars, part, recv, total;
  // direct: one unit stream per tile group in a cluster of one; each warp's rows are complete
  // and go straight to the output, so there are no partials.
  __host__ __device__ SwaSmem(int nw, int nst, int NT, int cs, int rows_pad, bool direct) {
    bars = (size_t)nw * nst * kStg;
    part = (bars + 8 * ((size_t)nw * nst + 1) + 15) / 16 * 16;
    recv = part + (direct ? 0 : (size_t)nw * NT * 8 * kRedStride * 4);
    total = recv + (size_t)(cs - 1) * rows_pad * kRedStride * 4;
  }
};

// Cluster plan: the ring's units over the warps of one cluster per (sequence, KV head).
SwaPlan make_plan(int cap, int S, int Hq, int Hkv) {
  SwaPlan pl{};
  const int nunits = cap / kUnit;
  const int R = S * (Hq / Hkv);
  const int ntiles = (R + 7) / 8;
  if (ntiles <= 3) {
    pl.NT = ntiles;
    pl.ntg = 1;
  } else {
    pl.NT = (ntiles + 1) / 2;
    pl.ntg = 2;
  }
  pl.rows_pad = pl.ntg * pl.NT * 8;
  const int nws_max = std::min(std::min(KVQ_SWA_STREAMS, kMaxStreams), 256 / (32 * pl.ntg));
  for (int nws = nws_max; nws >= 1; --nws) {
    pl.nws = nws;
    pl.cs = std::min(kMaxCluster, (nunits + nws - 1) / nws);
    const int ns = pl.cs * nws;
    pl.ups = (nunits + ns - 1) / ns;
    for (pl.nst = std::min(2, pl.ups); pl.nst >= 1; --pl.nst) {
      pl.smem = SwaSmem(nws * pl.ntg, pl.nst, pl.NT, pl.cs, pl.rows_pad, nws == 1 && pl.cs == 1).total;
      if (pl.smem <= kSmemCap) return pl;
    }
  }
  pl.smem = 0;  // does not fit (40 or more query rows per KV head): the split-K path
  return pl;
}

// Output dim of accumulator row `row` (0..15) of PV m-tile `mt` (0..7): m-tile mt covers the
// 16 dims 16 mt .. 16 mt + 15, its row r holding dim 16 mt + 2 (r & 7) + (r >> 3) because V's
// e4m3 bytes are split into even/odd dims by the byte permute before conversion.
__device__ __forceinline__ int swa_out_dim(int mt, int row) { return 16 * mt + 2 * (row & 7) + (row >> 3); }

// Byte offset of lane l's four codes of the record in ring slot `slot` within a unit's K (or
// V) records: same chunk order as in the ring block (chunk c at c ^ (slot & 7)).
__device__ __forceinline__ int unit_lane_offset(int slot, int lane) {
  return (slot & (kUnit - 1)) * kRec8 + ((lane >> 2) ^ (slot & 7)) * 16 + ((4 * lane) & 15);
}

// One 32-slot unit (K records then V records at `st`, unit index u) against the warp's query tiles.
template <int NT>
__device__ __forceinline__ void attend_unit(const uint8_t* st, int u, int p_last, int slot_last, int cap,
                                            float score_scale, const uint32_t (&qf)[NT][8][2],
                                            const int (&lim_lo)[NT][2], const int (&lim_hi)[NT][2],
                                            float (&m)[NT][2], float (&l)[NT][2], float (&acc)[NT][8][4],
                                            int lane) {
  const int g = lane >> 2, t = lane & 3;
  // ---- scores: S[slot][row] = sum_d K[slot][d] q[row][d], K and q in f16 (exact for e4m3)
  float sc[NT][2][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    float d[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) d[nt][c] = 0.0f;
    const int ta = 16 * mt + g, tb = ta + 8;  // both slots have (slot & 7) == g
    const uint4 a0 = *reinterpret_cast<const uint4*>(st + ta * kRec8 + 16 * ((2 * t) ^ g));
    const uint4 a1 = *reinterpret_cast<const uint4*>(st + ta * kRec8 + 16 * ((2 * t + 1) ^ g));
    const uint4 b0 = *reinterpret_cast<const uint4*>(st + tb * kRec8 + 16 * ((2 * t) ^ g));
    const uint4 b1 = *reinterpret_cast<const uint4*>(st + tb * kRec8 + 16 * ((2 * t + 1) ^ g));
    const uint32_t A[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t Bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t x0 = e4m3x2_to_f16x2(A[ks] & 0xFFFFu), x2 = e4m3x2_to_f16x2(A[ks] >> 16);
      const uint32_t x1 = e4m3x2_to_f16x2(Bw[ks] & 0xFFFFu), x3 = e4m3x2_to_f16x2(Bw[ks] >> 16);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816(d[nt], x0, x1, x2, x3, qf[nt][ks][0], qf[nt][ks][1]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) sc[nt][mt][c] = d[nt][c] * score_scale;
  }
  // ---- window mask: slot -> position through the newest slot
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int slot = u * kUnit + 16 * mt + g + 8 * hh;
      int back = slot_last - slot;
      if (back < 0) back += cap;
      const int pos = p_last - back;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
          if (pos < lim_lo[nt][jj] || pos > lim_hi[nt][jj]) sc[nt][mt][2 * hh + jj] = -INFINITY;
    }
  // ---- online softmax
  float muse[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      float mx = fmaxf(fmaxf(sc[nt][0][jj], sc[nt][0][2 + jj]), fmaxf(sc[nt][1][jj], sc[nt][1][2 + jj]));
      mx = warp_max_g(mx);
      const float mnew = fmaxf(m[nt][jj], mx);
      muse[nt][jj] = mnew == -INFINITY ? 0.0f : mnew;
      const float alpha = fast_exp2(m[nt][jj] - muse[nt][jj]);
      m[nt][jj] = mnew;
      if (alpha != 1.0f) {
        l[nt][jj] *= alpha;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[nt][i][jj] *= alpha;
          acc[nt][i][2 + jj] *= alpha;
        }
      }
    }
  // ---- P (transposed into a B fragment) and PV
  const uint8_t* Vs = st + kHalf;
  const int qi = lane >> 3, r8 = lane & 7;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float pr[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) pr[c] = fast_exp2(sc[nt][mt][c] - muse[nt][c & 1]);
      l[nt][0] += pr[0] + pr[2];
      l[nt][1] += pr[1] + pr[3];
      pb[nt][0] = movmatrix_trans(pack_f16x2(pr[0], pr[1]));
      pb[nt][1] = movmatrix_trans(pack_f16x2(pr[2], pr[3]));
    }
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int cprime = 2 * cc + (qi >> 1), th = qi & 1;
      const int slot = 16 * mt + 8 * th + r8;
      uint32_t rr[4];
      ldsm_x4_trans(rr, smem_addr(Vs + slot * kRec8 + 16 * (cprime ^ r8)));
#pragma unroll
      for (int ci = 0; ci < 2; ++ci) {
        const uint32_t y0 = prmt(rr[2 * ci], 0u, 0x3120u);
        const uint32_t y1 = prmt(rr[2 * ci + 1], 0u, 0x3120u);
        const uint32_t v0 = e4m3x2_to_f16x2(y0 & 0xFFFFu), v1 = e4m3x2_to_f16x2(y0 >> 16);
        const uint32_t v2 = e4m3x2_to_f16x2(y1 & 0xFFFFu), v3 = e4m3x2_to_f16x2(y1 >> 16);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816(acc[nt][2 * cc + ci], v0, v1, v2, v3, pb[nt][0], pb[nt][1]);
      }
    }
  }
}

// Issues the two bulk copies of unit u of this (sequence, KV head) into stage `st`.
__device__ __forceinline__ void load_unit(uint8_t* st, const uint8_t* seg, int u, uint64_t* bar, uint64_t pol) {
  const uint8_t* blk = seg + (size_t)(u >> 1) * kBlk + (u & 1) * kHalf;
  mbar_arrive_expect_tx(bar, kStg);
  bulk_g2s(st, blk, kHalf, bar, pol);
  bulk_g2s(st + kHalf, blk + kPage * kRec8, kHalf, bar, pol);
}

// Whether unit u holds a window position: a slot at most span back from slot_last (its slot
// nearest behind slot_last is d slots back, 0 if it holds slot_last).
__device__ __forceinline__ bool unit_in_window(int u, int slot_last, int span, int cap) {
  const int first = u * kUnit, last = first + kUnit - 1;
  const int d = (slot_last >= first && slot_last <= last) ? 0 : (slot_last - last + cap) % cap;
  return d <= span;
}

// Position word read without ordering against other grids (relaxed): a hint for prefetches
// issued before the grid wait; what the kernel uses is read again after it.
__device__ __forceinline__ int ld_relaxed_s32(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

template <int NT>
__global__ void __launch_bounds__(256, 1) swa_cluster_kernel(const SwaParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int nw = p.nws * p.ntg;
  const int ws = warp / p.ntg, tg = warp - (warp / p.ntg) * p.ntg;
  const int rank = (int)cluster_ctarank();
  const int pair = blockIdx.x / p.cs;  // (sequence, KV head) of this cluster
  const int b = pair / p.Hkv, h = pair - (pair / p.Hkv) * p.Hkv;
  const int stream = rank * p.nws + ws, nstream = p.cs * p.nws;
  const int nu = stream < p.nunits ? (p.nunits - 1 - stream) / nstream + 1 : 0;  // units of this stream
  const SwaSmem L(nw, p.nst, NT, p.cs, p.rows_pad, p.nws == 1 && p.cs == 1);
  uint8_t* wst = smem + (size_t)warp * p.nst * kStg;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* wfull = bars + warp * p.nst;
  uint64_t* recv_bar = bars + nw * p.nst;
  float* part = reinterpret_cast<float*>(smem + L.part);
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  uint8_t* seg = const_cast<uint8_t*>(p.ring) + (size_t)pair * p.nblk * kBlk;

  // ---- prologue, which may overlap the previous grid on the stream: barriers, and L2
  // prefetches of this stream's units and of the query and appended rows (L2 is coherent,
  // so a grid still writing them cannot leave stale copies). Nothing is read before
  // griddep_wait().
  const size_t rb = (size_t)kD * (p.bf16 ? 2 : 4);  // bytes per q / k / v row
  if (lane == 0) {
    for (int s = 0; s < p.nst; ++s) mbar_init(&wfull[s], 1);
    if (warp == 0) {
      mbar_init(recv_bar, 1);
      if (rank == 0) mbar_arrive_expect_tx(recv_bar, (uint32_t)((p.cs - 1) * p.R * kPushBytes));
    }
    fence_barrier_init();
    fence_proxy_async_shared();
    // the units copied first (all of a cluster plan's); a one-CTA plan (many sequences) copies
    // units that hold window positions once the position is known, so it prefetches the first of
    // those as the position hint places them
    if (tg == 0 && p.cs > 1) {
      for (int i = 0; i < min(nu, 2 * p.nst); ++i) {
        const int u = stream + i * nstream;
        const uint8_t* blk = seg + (size_t)(u >> 1) * kBlk + (u & 1) * kHalf;
        prefetch_l2_bulk(blk, kHalf);
        prefetch_l2_bulk(blk + kPage * kRec8, kHalf);
      }
    } else if (tg == 0) {
      const int ch = max(0, ld_relaxed_s32(p.pos0 + b));
      const int pl = ch + p.S - 1, sl = pl % p.cap, sp = pl - max(0, ch - p.window + 1);
      for (int i = 0, n = 0; i < nu && n < 2 * p.nst; ++i) {
        const int u = stream + i * nstream;
        if (!unit_in_window(u, sl, sp, p.cap)) continue;
        const uint8_t* blk = seg + (size_t)(u >> 1) * kBlk + (u & 1) * kHalf;
        prefetch_l2_bulk(blk, kHalf);
        prefetch_l2_bulk(blk + kPage * kRec8, kHalf);
        ++n;
      }
    }
    if (warp == 0 && rank == 0) {
      prefetch_l2(p.pos0 + b);
      for (int r = 0; r < p.S; ++r)  // the G query rows of this KV head are contiguous
        prefetch_l2_bulk(static_cast<const uint8_t*>(p.q) + (((size_t)b * p.S + r) * p.Hq + (size_t)h * p.G) * rb,
                         (uint32_t)(p.G * rb));
    }
  }
  if (p.k_new != nullptr && warp == 0 && lane < 2 * p.S) {
    const size_t row = ((size_t)b * p.S + (lane >> 1)) * p.Hkv + h;
    prefetch_l2_bulk(static_cast<const uint8_t*>((lane & 1) ? p.v_new : p.k_new) + row * rb, (uint32_t)rb);
  }
  __syncwarp();
  cluster_arrive_relaxed();
  griddep_wait();
  griddep_launch_dependents();  // after the wait: at most one grid runs ahead

  // ---- this warp's first copies (L2 hits when the prefetch had time to land); a one-CTA plan
  // copies once the position is known (just below)
  if (p.cs > 1 && lane == 0) {
    const uint64_t pol = policy_evict_first();
    for (int i = 0; i < min(p.nst, nu); ++i)
      load_unit(wst + (size_t)i * kStg, seg, stream + i * nstream, &wfull[i], pol);
  }
  __syncwarp();

  // Every load below is issued before any result is used: the first position, the query rows
  // and the first appended key/value row (S = 1 decode appends one; its owner is known only
  // once the position is, so every warp loads it). No atomic sits between them, so the loads
  // need not wait for a branch on the position.
  const int c0raw = p.pos0[b];
  float xnew[2][4];  // appended row r = 0: key, value
  if (p.k_new != nullptr) {
    const size_t row0 = (size_t)b * p.S * p.Hkv + h;
    load_row4(p.k_new, p.bf16, row0, lane, xnew[0]);
    load_row4(p.v_new, p.bf16, row0, lane, xnew[1]);
  }

  int c0 = c0raw;
  if (c0 < 0) {
    if (rank == 0 && threadIdx.x == 0) set_err(p.dev_err, KVQ_DEVERR_POS);
    c0 = 0;
  }
  const int p_last = c0 + p.S - 1;  // newest position after the append
  const int slot_last = p_last % p.cap;

  const int span = p_last - max(0, c0 - p.window + 1);
  int issued = p.cs > 1 ? min(p.nst, nu) : 0;  // units issued so far (warp-uniform)
  int next_i = issued;          // the stream's next unit index to consider for a refill
  int su0 = stream, su1 = stream + nstream;  // unit held by stage 0 / 1 (nst <= 2)
  int done = 0;                 // units consumed
  // the stream's next unit that holds a window position
  auto next_window_unit = [&]() {
    for (; next_i < nu; ++next_i)
      if (unit_in_window(stream + next_i * nstream, slot_last, span, p.cap)) break;
  };
  if (p.cs == 1) {  // the first copies, now that the window is known
    for (int s = 0; s < p.nst; ++s) {
      next_window_unit();
      if (next_i >= nu) break;
      const int un = stream + next_i * nstream;
      if (lane == 0) load_unit(wst + (size_t)s * kStg, seg, un, &wfull[s], policy_evict_first());
      if (s == 0) su0 = un;
      else su1 = un;
      ++next_i;
      ++issued;
    }
  }
  // ---- query fragments (B operand, 8 rows per tile)
  uint32_t qf[NT][8][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tile = tg * NT + nt;
    const int nB = 8 * tile + g;
    float qv[32];
    if (nB < p.R) {
      const size_t row = ((size_t)b * p.S + nB / p.G) * p.Hq + h * p.G + nB % p.G;
      if (!p.bf16) {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.q) + row * kD + 32 * t);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 v = src[i];
          qv[4 * i] = v.x;
          qv[4 * i + 1] = v.y;
          qv[4 * i + 2] = v.z;
          qv[4 * i + 3] = v.w;
        }
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) + row * kD + 32 * t);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = src[i];
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            qv[8 * i + 2 * k] = bf16_bits_to_f32(w[k] & 0xFFFFu);
            qv[8 * i + 2 * k + 1] = bf16_bits_to_f32(w[k] >> 16);
          }
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) qv[i] = 0.0f;
    }
    // k-step ks covers dims 32 t' + 4 ks .. +3 of lane t' (the K words are read in the
    // matching order, so the dot product pairs every dim with itself)
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qf[nt][ks][0] = pack_f16x2(qv[4 * ks], qv[4 * ks + 1]);
      qf[nt][ks][1] = pack_f16x2(qv[4 * ks + 2], qv[4 * ks + 3]);
    }
  }

  // ---- per-row window limits
  int lim_lo[NT][2], lim_hi[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int nC = 8 * (tg * NT + nt) + 2 * t + jj;
      const int r = nC < p.R ? nC / p.G : 0;
      lim_hi[nt][jj] = c0 + r;
      lim_lo[nt][jj] = max(0, c0 + r - p.window + 1);
    }
  }

  // ---- appended rows that fall in this stream's units: encode now (the loads overlap the copies)
  uint32_t code[8][2];
  uint32_t have = 0;  // bit 2 r + which: code[r][which] is valid and belongs to one of my units
  if (p.k_new != nullptr) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      code[r][0] = code[r][1] = 0;
      if (r >= p.S) continue;
      const int slot = (c0 + r) % p.cap;
      const int u = slot / kUnit;
      if (u < stream || (u - stream) % nstream != 0) continue;
      const size_t row = ((size_t)b * p.S + r) * p.Hkv + h;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        float x[4];
        if (r == 0) {
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] = xnew[which][e];
        } else {
          load_row4(which ? p.v_new : p.k_new, p.bf16, row, lane, x);
        }
        if (!warp_all_finite(x)) {
          if (lane == 0 && tg == 0) set_err(p.dev_err, KVQ_DEVERR_NONFINITE);
          continue;
        }
        code[r][which] = fp8_encode4(x, which ? p.v_scale : p.k_scale);
        have |= 1u << (2 * r + which);
        if (tg == 0)  // the ring copy for later steps, written once per unit
          *reinterpret_cast<uint32_t*>(seg + (size_t)(slot / kPage) * kBlk + which * kPage * kRec8 +
                                       fp8_lane_offset(slot, lane)) = code[r][which];
      }
    }
  }

  float m[NT][2], l[NT][2], acc[NT][8][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      m[nt][jj] = -INFINITY;
      l[nt][jj] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[nt][i][c] = 0.0f;
  }

  // Units are consumed in the order they were issued. A cluster plan's first min(nst, nu) are the
  // stream's first units, copied before the position was known; a one-CTA plan's first ones, and
  // every refill, are the stream's next units that hold a position of the rows' windows
  // [max(0, c0 - window + 1), p_last]: units wholly outside them (the ring's slots beyond the
  // window, and slots not yet written) are skipped. A unit holding an appended row is never
  // skipped.
  for (int k = 0; k < issued; ++k) {
    const int s = k % p.nst;
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&wfull[s], (uint32_t)(k / p.nst) & 1u));
    if (!ok) {
      if (lane == 0) set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
      break;
    }
    uint8_t* st = wst + (size_t)s * kStg;
    const int u = s == 0 ? su0 : su1;
    if (have) {
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (r >= p.S) break;
        const int slot = (c0 + r) % p.cap;
        if (slot / kUnit != u) continue;
#pragma unroll
        for (int which = 0; which < 2; ++which)
          if (have >> (2 * r + which) & 1u)
            *reinterpret_cast<uint32_t*>(st + which * kHalf + unit_lane_offset(slot, lane)) = code[r][which];
      }
      __syncwarp();
    }
    attend_unit<NT>(st, u, p_last, slot_last, p.cap, p.score_scale, qf, lim_lo, lim_hi, m, l, acc, lane);
    done = k + 1;
    __syncwarp();
    // refill this stage with the stream's next unit that holds a window position
    next_window_unit();
    if (next_i < nu) {
      const int un = stream + next_i * nstream;
      if (lane == 0) {
        fence_proxy_async_shared();
        load_unit(st, seg, un, &wfull[s], policy_evict_first());
      }
      if (s == 0) su0 = un;
      else su1 = un;
      ++next_i;
      ++issued;
    }
  }
  if (done < issued && lane == 0) {  // gave up: let the copies still in flight land before leaving
    for (int k = done; k < min(issued, done + p.nst); ++k)
      if (!mbar_wait_bounded(&wfull[k % p.nst], (uint32_t)(k / p.nst) & 1u)) break;
  }

  if (p.nws == 1 && p.cs == 1) {
    // ---- the only stream of this tile group: its rows are complete; normalise and store them
    // (lane: dims 16 i + 2 g and 16 i + 2 g + 1 of rows 2 t and 2 t + 1 of each tile)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const float lt = warp_sum_g(l[nt][jj]);
        const int row = (tg * NT + nt) * 8 + 2 * t + jj;
        if (row < p.R) {
          const float inv = 1.0f / lt;
          const int r = row / p.G, gi = row - (row / p.G) * p.G;
          float* dst = p.out + (((size_t)b * p.S + r) * p.Hq + h * p.G + gi) * kD + 2 * g;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float2*>(dst + 16 * i) =
                make_float2(acc[nt][i][jj] * p.v_scale * inv, acc[nt][i][2 + jj] * p.v_scale * inv);
        }
      }
    }
    cluster_wait();
    return;
  }

  // ---- this stream's partial for its tile group's rows
  float* mypart = part + (size_t)warp * NT * 8 * kRedStride;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const float lt = warp_sum_g(l[nt][jj]);
      float* dst = mypart + (8 * nt + 2 * t + jj) * kRedStride;
      if (g == 0) {
        dst[0] = m[nt][jj];
        dst[1] = lt;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        dst[4 + swa_out_dim(i, g)] = acc[nt][i][jj] * p.v_scale;
        dst[4 + swa_out_dim(i, g + 8)] = acc[nt][i][2 + jj] * p.v_scale;
      }
    }
  }
  __syncthreads();
  cluster_wait();  // CTA 0's receive barrier is initialised and armed

  // ---- merge: item = (query row, 8 consecutive dims). Every CTA merges its own streams; the
  // other CTAs push that into CTA 0, which merges the cluster and writes the output.
  const uint32_t bar0 = map_cluster(smem_addr(recv_bar), 0);
  const uint32_t recv0 = map_cluster(smem_addr(recv), 0);
  bool received = false;  // CTA 0: the other CTAs' pushes have landed (waited after the own merge)
  for (int e = threadIdx.x; e < p.R * 16; e += blockDim.x) {
    const int row = e >> 4, c8 = e & 15;
    const int tgr = (row >> 3) / NT;  // tile group holding this row
    const int rl = row - 8 * NT * tgr;
    float mk[kMaxStreams];
#pragma unroll
    for (int w2 = 0; w2 < kMaxStreams; ++w2)
      mk[w2] = w2 < p.nws ? part[((size_t)(w2 * p.ntg + tgr) * NT * 8 + rl) * kRedStride] : -INFINITY;
    float M = mk[0];
#pragma unroll
    for (int w2 = 1; w2 < kMaxStreams; ++w2) M = fmaxf(M, mk[w2]);
    const float Mu = M == -INFINITY ? 0.0f : M;
    float lsum = 0.0f;
    float a[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int w2 = 0; w2 < kMaxStreams; ++w2) {
      if (w2 >= p.nws) break;
      const float* src = part + ((size_t)(w2 * p.ntg + tgr) * NT * 8 + rl) * kRedStride;
      const float wgt = fast_exp2(mk[w2] - Mu);
      const float4 v0 = reinterpret_cast<const float4*>(src + 4)[2 * c8];
      const float4 v1 = reinterpret_cast<const float4*>(src + 4)[2 * c8 + 1];
      lsum = fmaf(wgt, src[1], lsum);
      a[0] = fmaf(wgt, v0.x, a[0]);
      a[1] = fmaf(wgt, v0.y, a[1]);
      a[2] = fmaf(wgt, v0.z, a[2]);
      a[3] = fmaf(wgt, v0.w, a[3]);
      a[4] = fmaf(wgt, v1.x, a[4]);
      a[5] = fmaf(wgt, v1.y, a[5]);
      a[6] = fmaf(wgt, v1.z, a[6]);
      a[7] = fmaf(wgt, v1.w, a[7]);
    }
    if (rank != 0) {
      const uint32_t dst = recv0 + 4u * (uint32_t)(((rank - 1) * p.rows_pad + row) * kRedStride);
      if (c8 == 0) st_async_f32x2(dst, M, lsum, bar0);
      st_async_f32x4(dst + 16 + 32 * c8, make_float4(a[0], a[1], a[2], a[3]), bar0);
      st_async_f32x4(dst + 32 + 32 * c8, make_float4(a[4], a[5], a[6], a[7]), bar0);
      continue;
    }
    // CTA 0: fold in the other CTAs' partials (relative to their own maxima). Threads with an
    // item wait for the pushes, so the CTA outlives the copies into its shared memory.
    if (!received) {
      if (!mbar_wait_bounded(recv_bar, 0)) set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
      received = true;
    }
    float mr[kMaxCluster];
    float Mc = M;
#pragma unroll
    for (int rr = 1; rr < kMaxCluster; ++rr) {
      mr[rr] = rr < p.cs ? recv[((rr - 1) * p.rows_pad + row) * kRedStride] : -INFINITY;
      Mc = fmaxf(Mc, mr[rr]);
    }
    const float Mcu = Mc == -INFINITY ? 0.0f : Mc;
    const float w0 = fast_exp2(M - Mcu);
    lsum *= w0;
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] *= w0;
#pragma unroll
    for (int rr = 1; rr < kMaxCluster; ++rr) {
      if (rr >= p.cs) break;
      const float* sr = recv + ((rr - 1) * p.rows_pad + row) * kRedStride;
      const float wgt = fast_exp2(mr[rr] - Mcu);
      const float4 v0 = reinterpret_cast<const float4*>(sr + 4)[2 * c8];
      const float4 v1 = reinterpret_cast<const float4*>(sr + 4)[2 * c8 + 1];
      lsum = fmaf(wgt, sr[1], lsum);
      a[0] = fmaf(wgt, v0.x, a[0]);
      a[1] = fmaf(wgt, v0.y, a[1]);
      a[2] = fmaf(wgt, v0.z, a[2]);
      a[3] = fmaf(wgt, v0.w, a[3]);
      a[4] = fmaf(wgt, v1.x, a[4]);
      a[5] = fmaf(wgt, v1.y, a[5]);
      a[6] = fmaf(wgt, v1.z, a[6]);
      a[7] = fmaf(wgt, v1.w, a[7]);
    }
    const int r = row / p.G, gi = row - (row / p.G) * p.G;
    const float inv = 1.0f / lsum;
    float4* dst = reinterpret_cast<float4*>(p.out + (((size_t)b * p.S + r) * p.Hq + h * p.G + gi) * kD) + 2 * c8;
    dst[0] = make_float4(a[0] * inv, a[1] * inv, a[2] * inv, a[3] * inv);
    dst[1] = make_float4(a[4] * inv, a[5] * inv, a[6] * inv, a[7] * inv);
  }
}

struct SwaDevCache {
  bool attr[4] = {false};
  int sm = 0;
  int occ[4][3][kMaxStreams + 1][KVQ_SWA_BATCH_STAGES + 1] = {};  // resident CTAs per SM by [NT][ntg][nws][nst]
};
SwaDevCache g_swa_dev[64];
std::mutex g_swa_mu;  // guards g_swa_dev

SwaDevCache& dev_cache(int dev) { return g_swa_dev[(dev >= 0 && dev < 64) ? dev : 0]; }

// Call with g_swa_mu held: allow the kernel its dynamic shared memory (once per device).
template <int NT>
cudaError_t ensure_attr(SwaDevCache& dc) {
  if (dc.attr[NT]) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(swa_cluster_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemCap);
  if (e == cudaSuccess) dc.attr[NT] = true;
  return e;
}

template <int NT>
cudaError_t launch_swa_t(const SwaParams& p, size_t smem, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(g_swa_mu);
    const cudaError_t e = ensure_attr<NT>(dev_cache(dev));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)((long long)p.B * p.Hkv * p.cs), 1, 1);
  cfg.blockDim = dim3((unsigned)(p.nws * p.ntg * 32), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // the prologue (barriers, L2 prefetches) may overlap the previous grid on the stream
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, swa_cluster_kernel<NT>, p);
}

template <int NT>
int occupancy_t(int threads, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, swa_cluster_kernel<NT>, threads, smem) != cudaSuccess)
    return 0;
  return n;
}

struct DeviceShape {
  int dev, sm;
};

// Current device and its SM count (sm = 0 if it cannot be read: then only the cluster plans apply).
DeviceShape device_shape() {
  DeviceShape d{0, 0};
  if (cudaGetDevice(&d.dev) != cudaSuccess) return d;
  std::lock_guard<std::mutex> lock(g_swa_mu);
  SwaDevCache& dc = dev_cache(d.dev);
  if (dc.sm == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d.dev) != cudaSuccess) return d;
    dc.sm = n;
  }
  d.sm = dc.sm;
  return d;
}

// Resident one-CTA-per-pair CTAs per SM for this plan shape (0 if unknown).
int ctas_per_sm(int dev, const SwaPlan& pl) {
  std::lock_guard<std::mutex> lock(g_swa_mu);
  SwaDevCache& dc = dev_cache(dev);
  int& o = dc.occ[pl.NT][pl.ntg][pl.nws][pl.nst];
  if (o == 0) {
    const int threads = pl.nws * pl.ntg * 32;
    cudaError_t e;
    switch (pl.NT) {
      case 1: e = ensure_attr<1>(dc); o = e == cudaSuccess ? occupancy_t<1>(threads, pl.smem) : 0; break;
      case 2: e = ensure_attr<2>(dc); o = e == cudaSuccess ? occupancy_t<2>(threads, pl.smem) : 0; break;
      default: e = ensure_attr<3>(dc); o = e == cudaSuccess ? occupancy_t<3>(threads, pl.smem) : 0; break;
    }
  }
  return o;
}

// The plan for a call. With at least as many (sequence, KV head) pairs as SMs the pairs fill
// the GPU unsplit: one CTA per pair, its units over nws streams. The grid then runs in
// ceil(pairs / (SMs x resident CTAs)) waves of up to ceil(units / nws) units per stream; nws
// takes the fewest waves, then the fewest units per stream (a later wave of CTAs costs more
// than longer streams in one), then the fewest streams. With fewer pairs the cluster plan.
SwaPlan choose_plan(int cap, int B, int S, int Hq, int Hkv) {
  const SwaPlan cl = make_plan(cap, S, Hq, Hkv);
  const long long pairs = (long long)B * Hkv;
  const DeviceShape d = device_shape();
  if (d.sm <= 0 || pairs < d.sm) return cl;
  const int nunits = cap / kUnit;
  const int nws_max = std::min(std::min(KVQ_SWA_STREAMS, kMaxStreams), 256 / (32 * cl.ntg));
  SwaPlan best{};
  long long best_cost = -1;
  for (int nws = 1; nws <= nws_max; ++nws) {
    SwaPlan pl = cl;
    pl.nws = nws;
    pl.cs = 1;
    pl.ups = (nunits + nws - 1) / nws;
    if (pl.ups > kMaxUnitsBatched) continue;
    pl.batched = true;
    pl.smem = 0;
    for (pl.nst = std::min(KVQ_SWA_BATCH_STAGES, pl.ups); pl.nst >= 1; --pl.nst) {
      const size_t bytes = SwaSmem(nws * pl.ntg, pl.nst, pl.NT, 1, pl.rows_pad, nws == 1).total;
      if (bytes <= kSmemCap) {
        pl.smem = bytes;
        break;
      }
    }
    if (pl.smem == 0) continue;
    const int occ = ctas_per_sm(d.dev, pl);
    if (occ <= 0) continue;
    const long long slots = (long long)d.sm * occ;
    const long long cost = (pairs + slots - 1) / slots * 1000 + pl.ups;
    if (best_cost < 0 || cost < best_cost) {
      best = pl;
      best_cost = cost;
    }
  }
  return best_cost < 0 ? cl : best;
}

}  // namespace

bool swa_cluster_path(int capacity, int B, int S, int Hq, int Hkv) {
  const SwaPlan pl = choose_plan(capacity, B, S, Hq, Hkv);
  return pl.smem != 0 && (pl.batched || pl.ups <= kMaxUnitsPerStream);
}

void swa_plan_shape(int capacity, int B, int S, int Hq, int Hkv, int out[4]) {
  const SwaPlan pl = choose_plan(capacity, B, S, Hq, Hkv);
  const bool cluster = pl.smem != 0 && (pl.batched || pl.ups <= kMaxUnitsPerStream);
  out[0] = cluster ? pl.cs : 0;
  out[1] = cluster ? pl.nws : 0;
  out[2] = cluster ? pl.nst : 0;
  out[3] = cluster ? pl.ups : 0;
}

cudaError_t launch_swa_cluster(const AttnJob& job, cudaStream_t stream) {
  const SwaPlan pl = choose_plan(job.ring.capacity, job.B, job.S, job.Hq, job.Hkv);
  SwaParams p{};
  p.ring = job.ring.data;
  p.cap = job.ring.capacity;
  p.nblk = p.cap / kPage;
  p.nunits = p.cap / kUnit;
  p.window = job.window;
  p.B = job.B;
  p.S = job.S;
  p.Hq = job.Hq;
  p.Hkv = job.Hkv;
  p.G = job.Hq / job.Hkv;
  p.R = p.S * p.G;
  p.pos0 = job.ctx;
  p.q = job.q;
  p.bf16 = job.q_bf16;
  p.k_new = job.k_new;
  p.v_new = job.v_new;
  p.k_scale = job.k_scale;
  p.v_scale = job.v_scale;
  p.score_scale = job.sm_scale * kLog2e * job.k_scale;
  p.out = job.out;
  p.dev_err = job.dev_err;
  p.cs = pl.cs;
  p.nws = pl.nws;
  p.ntg = pl.ntg;
  p.nst = pl.nst;
  p.rows_pad = pl.rows_pad;
  switch (pl.NT) {
    case 1: return launch_swa_t<1>(p, pl.smem, stream);
    case 2: return launch_swa_t<2>(p, pl.smem, stream);
    default: return launch_swa_t<3>(p, pl.smem, stream);
  }
}

}  // namespace kvq
