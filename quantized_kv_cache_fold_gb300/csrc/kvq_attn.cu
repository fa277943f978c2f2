// Split-K flash-decoding attention over the rotated int4 cache and the FP8 ring.
//
// "Serving Kolibri-1 with a 4-bit KV cache", section "What we do": decode reads the 4-bit
// codes directly and nothing is rotated back. Sliding-window layers whose FP8 ring is too
// large for one thread-block cluster per (sequence, KV head) (kvq_swa.cu) read it through
// the same kernel (FMT = 1).
//
// Work split (stream-K over pages): every (sequence b, KV head h) is a segment of np_b
// pages; the segments are laid end to end and each CTA takes an equal contiguous range of
// pages, so ragged contexts balance to within one page. A CTA emits one partial
// (m, l, acc[128] per query row) for every segment it touches, into slot cta + segment;
// combine_kernel merges a segment's partials with log-sum-exp weights.
//
// Inside a CTA: one producer warp streams page-head blocks (K codes, V codes, K/V meta)
// into a ring of shared-memory stages with bulk asynchronous copies (TMA engine) signalled
// on mbarriers; consumer warps are arranged as token groups x tile groups. A tile is 8
// query rows (rows = S x G query heads of the KV head, row n = r*G + g). Per page a warp:
//   QK^T on tensor cores (mma.m16n8k16, fp32 accumulate): A = 16 tokens x 16 dims of K codes
//        read as the f16 subnormals c 2^-24 (low nibbles) or 16c 2^-24 (high nibbles, whose
//        query values are divided by 16), B = 16 dims x 8 query rows of q~ in f16, so the
//        accumulator holds 2^-24 sum q~ c up to fp32 rounding;
//   score = log2(e)*sm_scale*(s_K*dot + o_K*sum(q~)) -- scale and offset per token;
//   online softmax with exp2 against a lazily moved base (moved only when a score passes it
//        by more than 8, or by anything on pages with a V scale of 255 or more);
//   PV on tensor cores: A = 16 dims x 16 tokens of V codes read as f16 subnormals
//        (c - 7.5) 2^(k - 23), exact and centred (which keeps the fp32 sums of long contexts
//        small), B = 16 tokens x 8 rows of p*s_V in f16 (movmatrix transposes the QK
//        accumulator), plus sum_j p_j (o_V + 7.5 s_V) added per row; the partial undoes
//        2^(k - 23) per dim.

#include <algorithm>
#include <cmath>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

// Tuning of the attention CTA when one warp covers every query row of a KV head (S*G <= 8):
// consumer token groups, shared-memory pipeline stages and the register cap per thread.
#ifndef KVQ_TOKEN_GROUPS
#define KVQ_TOKEN_GROUPS 4
#endif
#ifndef KVQ_STAGES_INT4
#define KVQ_STAGES_INT4 12
#endif
#ifndef KVQ_INT4_MAXREG
#define KVQ_INT4_MAXREG 168
#endif
// int4 split kernel with 2 or 3 row tiles in one warp (one CTA per SM: about 250 registers a
// thread): 7 token groups, so 8 warps, two per SM sub-partition (4 -> 7: 300 -> 248 us at S = 2
// on the 64k workload), and 14 stages.
#ifndef KVQ_TILES3_TOKEN_GROUPS
#define KVQ_TILES3_TOKEN_GROUPS 7
#endif
#ifndef KVQ_TILES3_STAGES
#define KVQ_TILES3_STAGES 14
#endif
// 4 to 6 row tiles: two tile groups of up to 3 tiles, 3 token groups (7 warps), 6 stages.
#ifndef KVQ_TILES6_TOKEN_GROUPS
#define KVQ_TILES6_TOKEN_GROUPS 3
#endif
#ifndef KVQ_TILES6_STAGES
#define KVQ_TILES6_STAGES 6
#endif
// A consumer warp takes pages kg, kg + nkg, ... and page k lands in stage k mod nstages with
// phase parity (k / nstages) & 1. Parity only tells adjacent phases apart, so every stage
// must belong to one consumer warp (nstages a multiple of nkg); otherwise a warp running
// ahead could pass the wait for round f while round f - 1 of that stage is still in flight.
static_assert(KVQ_STAGES_INT4 % KVQ_TOKEN_GROUPS == 0, "stages must be a multiple of the token groups");

constexpr int kStage4 = 2 * kPage * kRec4 + 2 * kPage * 4;  // 8704 bytes: K codes, V codes, K meta, V meta
constexpr int kStage8 = 2 * kPage * kRec8;                  // 16384 bytes: K and V e4m3
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  // int4: page-head blocks [num_pages][Hkv][8704]; fp8: ring blocks [B][Hkv][cap/64][16384]
  const uint8_t* blocks;
  const int32_t* block_table;
  int max_pages;
  int num_pages;
  // fp8 ring
  int cap;
  int window;
  float v_scale;
  // shape
  int B, S, Hq, Hkv, G, R;
  const int32_t* ctx;
  const float* q_rot;
  const void* q;
  int q_bf16;
  float score_scale;
  float* partials;
  float* out;
  int32_t* dev_err;
  int ntg, nkg, nstages, rows_pad;
  int n_cta;
  // limit of the split kernel's waits on its shared-memory stages (consumers on a page's
  // copy, the producer on a stage's release); the drain of copies in flight keeps kWaitLimitNs
  unsigned long long stage_wait_ns;
};

__host__ __device__ __forceinline__ size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Per-lane online-softmax state of one 8-row tile as the token groups exchange it at a
// segment end: m and l and ov of the lane's two rows, then its 32 accumulator values.
constexpr int kMergeFloats = 6 + 32;

// Shared-memory layout, identical on host (sizing) and device.
struct SmemLayout {
  size_t stages, full, empty, valid, red, pre, flags, total;
  __host__ __device__ SmemLayout(int fmt, int nstages, int B, int nkg, int rows_pad) {
    const size_t stage = fmt == 0 ? kStage4 : kStage8;
    stages = 0;
    full = align_up(stages + nstages * stage, 16);
    empty = full + 8 * nstages;
    valid = empty + 8 * nstages;
    red = align_up(valid + 4 * nstages, 16);
    // one merge slot per tile group: kMergeFloats floats per lane per 8-row tile (lane-major)
    pre = align_up(red + (size_t)(rows_pad / 8) * kMergeFloats * 32 * 4, 128);
    flags = pre + 4 * (B + 1);
    total = align_up(flags + 16, 16);
  }
};

// Context length of sequence b as used by every kernel of one call (clamped into the
// cache; `bad` reports a clamp). Read at L2 (ld.global.cg): combine_kernel reads it before
// waiting for the previous grid, so no line an SM's L1 kept from an earlier call may serve it.
__device__ __forceinline__ int eff_ctx(const AttnParams& p, int b, bool& bad, int fmt) {
  int c = __ldcg(p.ctx + b);
  if (fmt == 0) {
    const int cap = p.max_pages * kPage - p.S;
    if (c < 0 || c > cap) {
      bad = true;
      c = min(max(c, 0), cap);
    }
  } else if (c < 0) {
    bad = true;
    c = 0;
  }
  return c;
}

__device__ __forceinline__ int seg_pages(const AttnParams& p, int ctxb, int fmt) {
  return fmt == 0 ? (ctxb + p.S + kPage - 1) / kPage : p.cap / kPage;
}

// Warp 0 builds pre[b] = sum_{b' < b} np_b' (pre[B] = total pages per KV head) and
// flags[1] = any clamped context. Other warps return at once.
__device__ void build_prefix(const AttnParams& p, int fmt, int* pre, volatile int* flags) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  if (fmt == 1) {  // every window segment spans the whole ring: no context lengths needed
    const int nblk = p.cap / kPage;
    for (int b = lane; b <= p.B; b += 32) pre[b] = b * nblk;
    if (lane == 0) {
      flags[0] = 0;
      flags[1] = 0;
    }
    return;
  }
  int carry = 0;
  bool bad = false;
  for (int base = 0; base < p.B; base += 32) {
    const int b = base + lane;
    int np = 0;
    if (b < p.B) np = seg_pages(p, eff_ctx(p, b, bad, fmt), fmt);
    int incl = np;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (b < p.B) pre[b] = carry + incl - np;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  const bool any_bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    pre[p.B] = carry;
    flags[0] = 0;
    flags[1] = any_bad ? 1 : 0;
  }
}

// Flattened page -> (sequence, head, local page, pages of the sequence).
__device__ __forceinline__ void decode_page(const int* pre, int B, int Hkv, long long pg, int& b, int& h, int& lp,
                                            int& np) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)Hkv * pre[mid] <= pg)
      lo = mid;
    else
      hi = mid - 1;
  }
  b = lo;
  np = pre[b + 1] - pre[b];
  // page of the sequence's head-major block: head = rem / np (< Hkv), by subtraction, which
  // keeps this inlined helper free of a 64-bit division
  long long rem = pg - (long long)Hkv * pre[b];
  int hh = 0;
  while (rem >= np) {
    rem -= np;
    ++hh;
  }
  h = hh;
  lp = (int)rem;
}

// CTA whose page range [floor(i P / n), floor((i+1) P / n)) contains page pg (n <= P).
__device__ __forceinline__ long long cta_of(long long pg, long long P, int n) { return ((pg + 1) * n - 1) / P; }

__device__ __forceinline__ float h2f_lo(uint32_t x) {
  return __half2float(__ushort_as_half((unsigned short)(x & 0xFFFFu)));
}
__device__ __forceinline__ float h2f_hi(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x >> 16))); }

// Output dim of accumulator row `row` (0..15) of PV m-tile `mt` (0..7).
template <int FMT>
__device__ __forceinline__ int out_dim(int mt, int row) {
  if (FMT == 0) return 32 * (mt >> 1) + 4 * (row & 7) + 2 * (mt & 1) + (row >> 3);
  return 16 * mt + 2 * (row & 7) + (row >> 3);
}

// Producer warp of the split kernels: the 32 lanes resolve the source blocks of 32 consecutive
// pages of the CTA's range [p0, p1) at once (block-table loads in parallel); lane 0 then issues
// one bulk copy per page into the ring of `nst` stages, in order, as stages free (`empty`, one
// phase per round), signalling `full`. A page whose block-table entry is out of range is
// flagged and delivered as invalid (valid[s] = 0, no copy). Waits for its own copies before
// returning.
template <int FMT>
__device__ __forceinline__ void produce_pages(const AttnParams& p, const int* pre, uint8_t* stages, uint64_t* full,
                                              uint64_t* empty, volatile int* valid, volatile int* flags, int nst,
                                              long long p0, long long p1, int lane) {
  constexpr int kStage = FMT == 0 ? kStage4 : kStage8;
  const uint64_t pol = policy_evict_first();
  const int npages = (int)(p1 - p0);
  int issued = 0;
  int s = 0, f = 0;  // stage and fill round of the next page
  for (int base = 0; base < npages; base += 32) {
    const int mine = base + lane;
    long long src = -1;  // byte offset of the page's block; -1 = invalid page
    if (mine < npages) {
      int b, h, lp, np;
      decode_page(pre, p.B, p.Hkv, p0 + mine, b, h, lp, np);
      if (FMT == 0) {
        const int phys = p.block_table[(size_t)b * p.max_pages + lp];
        if (phys >= 0 && phys < p.num_pages)
          src = ((long long)phys * p.Hkv + h) * kStage4;
        else
          set_err(p.dev_err, KVQ_DEVERR_PAGE);
      } else {
        src = (((long long)b * p.Hkv + h) * (p.cap / kPage) + lp) * kStage8;
      }
    }
    const int n = min(32, npages - base);
    int halt = 0;
    for (int j = 0; j < n; ++j) {
      const long long sj = __shfl_sync(0xffffffffu, src, j);
      if (lane == 0 && !halt) {
        if (f > 0 && !mbar_wait_bounded(&empty[s], (f - 1) & 1, p.stage_wait_ns)) {
          set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
          flags[0] = 1;
          halt = 1;
        } else {
          if (sj < 0) {
            valid[s] = 0;
            mbar_arrive(&full[s]);
          } else {
            valid[s] = 1;
            mbar_arrive_expect_tx(&full[s], kStage);
            bulk_g2s(stages + (size_t)s * kStage, p.blocks + sj, kStage, &full[s], pol);
          }
          ++issued;
          if (++s == nst) {
            s = 0;
            ++f;
          }
        }
      }
    }
    if (__shfl_sync(0xffffffffu, halt | flags[0], 0)) break;
  }
  // Do not retire while copies into this CTA's shared memory may be in flight.
  if (lane == 0) {
    for (int st = 0; st < nst && st < issued; ++st) {
      const int last = st + ((issued - 1 - st) / nst) * nst;
      if (!mbar_wait_bounded(&full[st], (last / nst) & 1)) set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
    }
  }
}

// Register caps: the int4 single-tile CTA (5 warps) must fit twice per SM, i.e. 3 warps per
// SM sub-partition -> at most 170 registers.
template <int FMT, int NT>
__global__ void __maxnreg__(NT == 1 ? (FMT == 0 ? KVQ_INT4_MAXREG : 184) : 255)
    attn_kernel(const AttnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kStage = FMT == 0 ? kStage4 : kStage8;
  constexpr int MTU = NT == 1 ? 4 : 2;  // 16-token m-tiles per online-softmax update
  const SmemLayout L(FMT, p.nstages, p.B, p.nkg, p.rows_pad);
  uint8_t* stages = smem + L.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
  volatile int* valid = reinterpret_cast<volatile int*>(smem + L.valid);
  int* pre = reinterpret_cast<int*>(smem + L.pre);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + L.flags);
  float* red = reinterpret_cast<float*>(smem + L.red);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwc = p.ntg * p.nkg;
  const int nst = p.nstages;

  // Launched with programmatic serialisation: the setup runs while the previous grid (the call's
  // prologue/append kernel, or the window append) finishes. It reads only context lengths (the
  // page prefix): no kernel of the call writes them, and the grids before the previous one
  // completed before this grid could launch. Everything after the setup waits for the previous
  // grid.
  build_prefix(p, FMT, pre, flags);
  if (threadIdx.x < nst) {
    mbar_init(&full[threadIdx.x], 1);
    mbar_init(&empty[threadIdx.x], p.ntg);
  }
  fence_barrier_init();
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();

  if (blockIdx.x == 0 && threadIdx.x == 0 && flags[1]) set_err(p.dev_err, KVQ_DEVERR_POS);
  const long long P = (long long)p.Hkv * pre[p.B];
  const int n_eff = (int)min((long long)p.n_cta, P);
  if ((int)blockIdx.x >= n_eff) return;
  const long long p0 = (long long)blockIdx.x * P / n_eff;
  const long long p1 = (long long)(blockIdx.x + 1) * P / n_eff;

  // ------------------------------------------------------------ producer warp
  if (warp == nwc) {
    produce_pages<FMT>(p, pre, stages, full, empty, valid, flags, nst, p0, p1, lane);
    return;
  }

  // ------------------------------------------------------------ consumer warps
  const int kg = warp / p.ntg, tg = warp - (warp / p.ntg) * p.ntg;
  const int g = lane >> 2, t = lane & 3;
  const int R = p.R, G = p.G;

  long long seg_start = p0;
  while (seg_start < p1) {
    int b, h, lp0, np;
    decode_page(pre, p.B, p.Hkv, seg_start, b, h, lp0, np);
    const long long seg_end = min(p1, seg_start + (np - lp0));
    const int seg = b * p.Hkv + h;
    bool bad_ctx = false;
    const int ctxb = eff_ctx(p, b, bad_ctx, FMT);
    if (FMT == 1 && bad_ctx && threadIdx.x == 0) set_err(p.dev_err, KVQ_DEVERR_POS);

    // ---- segment setup: query fragments and per-row limits
    uint32_t qf[NT][8][2];
    float qs[NT][2];
    int lim_lo[NT][2], lim_hi[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tile = tg * NT + nt;
      const int nB = 8 * tile + g;
      float qv[32];
      if (nB < R) {
        const size_t row = ((size_t)b * p.S + nB / G) * p.Hq + h * G + nB % G;
        if (FMT == 0 || !p.q_bf16) {
          const float* qbase = FMT == 0 ? p.q_rot : static_cast<const float*>(p.q);
          const float4* src = reinterpret_cast<const float4*>(qbase + row * kD + 32 * t);
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
      float part = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) part += qv[i];
      if (FMT == 0) {
        // k-step 2wi+e, slots (2t,2t+1) <- dims (8wi+2e, +4), slots (2t+8,2t+9) <- (+1, +5);
        // the second pair meets high nibbles, read as 16 c 2^-24 (unpack8_sub), so its query
        // values are divided by 16 (exact).
#pragma unroll
        for (int wi = 0; wi < 4; ++wi)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int d0 = 8 * wi + 2 * e;
            qf[nt][2 * wi + e][0] = pack_f16x2(qv[d0], qv[d0 + 4]);
            qf[nt][2 * wi + e][1] = pack_f16x2(qv[d0 + 1] * 0.0625f, qv[d0 + 5] * 0.0625f);
          }
      } else {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          qf[nt][ks][0] = pack_f16x2(qv[4 * ks], qv[4 * ks + 1]);
          qf[nt][ks][1] = pack_f16x2(qv[4 * ks + 2], qv[4 * ks + 3]);
        }
      }
      // full row sum (int4 offset term), then the sums of the rows of my accumulator columns
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float tot = __shfl_sync(0xffffffffu, part, (2 * t + j) * 4);
        qs[nt][j] = tot * p.score_scale;
        const int nC = 8 * tile + 2 * t + j;
        const int r = nC < R ? nC / G : 0;
        const int hi = ctxb + r;  // last visible position
        lim_hi[nt][j] = hi;
        lim_lo[nt][j] = FMT == 0 ? 0 : max(0, hi - p.window + 1);
      }
    }

    // Softmax state per accumulator row: m = exponent base (-inf until a finite score is seen),
    // muse = the base used in the exponent (0 while m is -inf), thr = how far a score may exceed
    // the base before it is moved (scores enter the exponent as s - muse).
    float m[NT][2], muse[NT][2], thr[NT][2], l[NT][2], ov[NT][2], acc[NT][8][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        m[nt][j] = -INFINITY;
        muse[nt][j] = 0.0f;
        thr[nt][j] = -INFINITY;
        l[nt][j] = 0.0f;
        ov[nt][j] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[nt][i][c] = 0.0f;
    }

    // fp8 ring: the newest position written and its slot
    const int p_last = ctxb + p.S - 1;
    const int slot_last = FMT == 1 ? p_last % p.cap : 0;

    const int k_beg = (int)(seg_start - p0), k_end = (int)(seg_end - p0);
    for (int k = k_beg + ((kg - k_beg % p.nkg + p.nkg) % p.nkg); k < k_end; k += p.nkg) {
      const long long pg = p0 + k;
      const int s = k % nst;
      const int f = k / nst;
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], f & 1, p.stage_wait_ns));
      if (!ok) {
        if (lane == 0) set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
        flags[0] = 1;
      }
      if (__any_sync(0xffffffffu, flags[0] != 0)) break;
      const int lp = lp0 + (int)(pg - seg_start);
      if (valid[s]) {
        const uint8_t* st = stages + (size_t)s * kStage;
        const bool need_mask = FMT == 1 || (lp + 1) * kPage > ctxb + 1;

#pragma unroll
        for (int mt0 = 0; mt0 < 4; mt0 += MTU) {
          // ---- per-token scale/offset (int4) for the tokens of this thread's accumulator rows
          float ka[MTU][2], kb[MTU][2], va[MTU][2], vb[MTU][2];
          if (FMT == 0) {
            const uint32_t* Km = reinterpret_cast<const uint32_t*>(st + 2 * kPage * kRec4);
            const uint32_t* Vm = Km + kPage;
#pragma unroll
            for (int u = 0; u < MTU; ++u)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int tok = 16 * (mt0 + u) + g + 8 * hh;
                const uint32_t mk = Km[tok], mv = Vm[tok];
                const float sk = h2f_lo(mk), ok_ = h2f_hi(mk), sv = h2f_lo(mv), ovv = h2f_hi(mv);
                ka[u][hh] = sk * p.score_scale * 16777216.0f;  // the MMA's products carry 2^-24
                kb[u][hh] = ok_;
                va[u][hh] = sv;
                vb[u][hh] = fmaf(7.5f, sv, ovv);
              }
          }

          // ---- scores
          float sc[NT][MTU][4];
          if (FMT == 0) {
            // Load every m-tile's K words first, then interleave the m-tiles' MMA chains so
            // independent accumulators hide the tensor-core latency.
            const uint8_t* Ks = st;
            uint32_t A[MTU][4], Bw[MTU][4];
#pragma unroll
            for (int u = 0; u < MTU; ++u) {
              // K record chunks sit at c ^ k_chunk_swz(slot): (g >> 1) & 1 for slot 16m + g, | 2 for + 8
              const int cw = 16 * (t ^ ((g >> 1) & 1));
              const uint4 wa = *reinterpret_cast<const uint4*>(Ks + (16 * (mt0 + u) + g) * kRec4 + cw);
              const uint4 wb = *reinterpret_cast<const uint4*>(Ks + (16 * (mt0 + u) + g + 8) * kRec4 + (cw ^ 32));
              A[u][0] = wa.x;
              A[u][1] = wa.y;
              A[u][2] = wa.z;
              A[u][3] = wa.w;
              Bw[u][0] = wb.x;
              Bw[u][1] = wb.y;
              Bw[u][2] = wb.z;
              Bw[u][3] = wb.w;
            }
            float d[NT][MTU][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int u = 0; u < MTU; ++u)
#pragma unroll
                for (int c = 0; c < 4; ++c) d[nt][u][c] = 0.0f;
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
              uint32_t ha[MTU][4], hb[MTU][4];
#pragma unroll
              for (int u = 0; u < MTU; ++u) {
                unpack8_sub(A[u][wi], ha[u]);
                unpack8_sub(Bw[u][wi], hb[u]);
              }
#pragma unroll
              for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int u = 0; u < MTU; ++u)
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt)
                    mma_16816(d[nt][u], ha[u][2 * e], hb[u][2 * e], ha[u][2 * e + 1], hb[u][2 * e + 1],
                              qf[nt][2 * wi + e][0], qf[nt][2 * wi + e][1]);
            }
#pragma unroll
            for (int u = 0; u < MTU; ++u)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  sc[nt][u][c] = fmaf(d[nt][u][c], ka[u][c >> 1], fmaf(kb[u][c >> 1], qs[nt][c & 1], -muse[nt][c & 1]));
          } else {
#pragma unroll
            for (int u = 0; u < MTU; ++u) {
              const int mt = mt0 + u;
              float d[NT][4];
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c) d[nt][c] = 0.0f;
              const uint8_t* Ks = st;
              const int ta = 16 * mt + g, tb = ta + 8;  // slot & 7 == g for both tokens
              const uint4 a0 = *reinterpret_cast<const uint4*>(Ks + ta * kRec8 + 16 * ((2 * t) ^ g));
              const uint4 a1 = *reinterpret_cast<const uint4*>(Ks + ta * kRec8 + 16 * ((2 * t + 1) ^ g));
              const uint4 b0 = *reinterpret_cast<const uint4*>(Ks + tb * kRec8 + 16 * ((2 * t) ^ g));
              const uint4 b1 = *reinterpret_cast<const uint4*>(Ks + tb * kRec8 + 16 * ((2 * t + 1) ^ g));
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
                for (int c = 0; c < 4; ++c)
                  sc[nt][u][c] = fmaf(d[nt][c], p.score_scale, -muse[nt][c & 1]);
            }
          }
          if (need_mask) {
#pragma unroll
            for (int u = 0; u < MTU; ++u)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int tok = 16 * (mt0 + u) + g + 8 * hh;
                int pos;
                if (FMT == 0) {
                  pos = lp * kPage + tok;
                } else {
                  const int slot = lp * kPage + tok;
                  int back = slot_last - slot;
                  if (back < 0) back += p.cap;
                  pos = p_last - back;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                  for (int j = 0; j < 2; ++j)
                    if (pos < lim_lo[nt][j] || pos > lim_hi[nt][j]) sc[nt][u][2 * hh + j] = -INFINITY;
              }
          }

          // ---- online softmax update
          // Lazy base: scores are already relative to muse. The base moves (to the running
          // maximum, rescaling l, ov and acc) only when some score of the page exceeds it by
          // more than 8, so P stays <= 2^8 and most pages skip the cross-lane maximum. P s_V
          // enters the PV product in f16, which stays finite for P <= 2^8 while s_V < 255; a page
          // holding a larger V scale moves the base as soon as any score exceeds it, so that
          // there P <= 1 and P s_V <= 65504.
          {
            float mx[NT][2];
            bool need = false;
            bool big = false;
            if (FMT == 0) {
              float vmax = 0.0f;
#pragma unroll
              for (int u = 0; u < MTU; ++u) vmax = fmaxf(vmax, fmaxf(va[u][0], va[u][1]));
              big = vmax >= 255.0f;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                float v = -INFINITY;
#pragma unroll
                for (int u = 0; u < MTU; ++u) v = fmaxf(v, fmaxf(sc[nt][u][j], sc[nt][u][2 + j]));
                mx[nt][j] = v;
                need |= v > (big ? fminf(thr[nt][j], 0.0f) : thr[nt][j]);
              }
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                  const float mt = warp_max_g(mx[nt][j]);
                  const float mnew = fmaxf(m[nt][j], muse[nt][j] + mt);
                  if (mnew != m[nt][j]) {
                    const float mu2 = mnew == -INFINITY ? 0.0f : mnew;
                    const float alpha = fast_exp2(m[nt][j] - mu2);
                    const float delta = muse[nt][j] - mu2;
                    l[nt][j] *= alpha;
                    ov[nt][j] *= alpha;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                      acc[nt][i][j] *= alpha;
                      acc[nt][i][2 + j] *= alpha;
                    }
#pragma unroll
                    for (int u = 0; u < MTU; ++u) {
                      sc[nt][u][j] += delta;
                      sc[nt][u][2 + j] += delta;
                    }
                    m[nt][j] = mnew;
                    muse[nt][j] = mu2;
                    thr[nt][j] = mnew == -INFINITY ? -INFINITY : 8.0f;
                  }
                }
            }
          }

          // ---- P and PV
#pragma unroll
          for (int u = 0; u < MTU; ++u) {
            const int mt = mt0 + u;
            uint32_t pb[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              float pr[4];
#pragma unroll
              for (int c = 0; c < 4; ++c) pr[c] = fast_exp2(sc[nt][u][c]);
              l[nt][0] += pr[0] + pr[2];
              l[nt][1] += pr[1] + pr[3];
              if (FMT == 0) {
                ov[nt][0] = fmaf(pr[0], vb[u][0], fmaf(pr[2], vb[u][1], ov[nt][0]));
                ov[nt][1] = fmaf(pr[1], vb[u][0], fmaf(pr[3], vb[u][1], ov[nt][1]));
                pb[nt][0] = movmatrix_trans(pack_f16x2_sat(pr[0] * va[u][0], pr[1] * va[u][0]));
                pb[nt][1] = movmatrix_trans(pack_f16x2_sat(pr[2] * va[u][1], pr[3] * va[u][1]));
              } else {
                pb[nt][0] = movmatrix_trans(pack_f16x2(pr[0], pr[1]));
                pb[nt][1] = movmatrix_trans(pack_f16x2(pr[2], pr[3]));
              }
            }
            const uint8_t* Vs = st + kPage * (FMT == 0 ? kRec4 : kRec8);
            const int qi = lane >> 3, r8 = lane & 7;
            if (FMT == 0) {
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                const int cprime = 2 * cc + (qi >> 1), th = qi & 1;
                const int tok = 16 * mt + 8 * th + r8;
                uint32_t rr[4];
                ldsm_x4_trans(rr, smem_addr(Vs + tok * kRec4 + 16 * (cprime ^ (r8 >> 1))));
#pragma unroll
                for (int ci = 0; ci < 2; ++ci) {
                  uint32_t h0[4], h1[4];
                  unpack8_v(rr[2 * ci], h0);
                  unpack8_v(rr[2 * ci + 1], h1);
#pragma unroll
                  for (int e1 = 0; e1 < 2; ++e1) {
                    const int mtd = 2 * (2 * cc + ci) + e1;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                      mma_16816(acc[nt][mtd], h0[2 * e1], h0[2 * e1 + 1], h1[2 * e1], h1[2 * e1 + 1], pb[nt][0],
                                pb[nt][1]);
                  }
                }
              }
            } else {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                const int cprime = 2 * cc + (qi >> 1), th = qi & 1;
                const int tok = 16 * mt + 8 * th + r8;
                uint32_t rr[4];
                ldsm_x4_trans(rr, smem_addr(Vs + tok * kRec8 + 16 * (cprime ^ r8)));
#pragma unroll
                for (int ci = 0; ci < 2; ++ci) {
                  const uint32_t y0 = prmt(rr[2 * ci], 0u, 0x3120u);
                  const uint32_t y1 = prmt(rr[2 * ci + 1], 0u, 0x3120u);
                  const uint32_t a0 = e4m3x2_to_f16x2(y0 & 0xFFFFu), a1 = e4m3x2_to_f16x2(y0 >> 16);
                  const uint32_t a2 = e4m3x2_to_f16x2(y1 & 0xFFFFu), a3 = e4m3x2_to_f16x2(y1 >> 16);
                  const int mtd = 2 * cc + ci;
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt) mma_16816(acc[nt][mtd], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                }
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- segment end: the token groups' states are merged pairwise, lane by lane (every token
    // group of a tile group holds the same rows and dims in the same fragment positions), from
    // the last token group down to group 0 through one shared slot per tile group; group 0 then
    // reduces l and the offset term over its lanes and writes the CTA partial.
    float* mslot = red + (size_t)tg * NT * kMergeFloats * 32;
    for (int kk = p.nkg - 1; kk >= 1; --kk) {
      if (kg == kk) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float* q = mslot + (size_t)nt * kMergeFloats * 32 + lane;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            q[32 * j] = m[nt][j];
            q[32 * (2 + j)] = l[nt][j];
            q[32 * (4 + j)] = ov[nt][j];
          }
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) q[32 * (6 + 4 * i + c)] = acc[nt][i][c];
        }
      }
      named_barrier(1, nwc * 32);
      if (kg == kk - 1) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float* q = mslot + (size_t)nt * kMergeFloats * 32 + lane;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float mo = q[32 * j];
            const float mn = fmaxf(m[nt][j], mo);
            const float mu = mn == -INFINITY ? 0.0f : mn;
            const float a = fast_exp2(m[nt][j] - mu), bo = fast_exp2(mo - mu);
            l[nt][j] = fmaf(l[nt][j], a, q[32 * (2 + j)] * bo);
            ov[nt][j] = fmaf(ov[nt][j], a, q[32 * (4 + j)] * bo);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              acc[nt][i][j] = fmaf(acc[nt][i][j], a, q[32 * (6 + 4 * i + j)] * bo);
              acc[nt][i][2 + j] = fmaf(acc[nt][i][2 + j], a, q[32 * (6 + 4 * i + 2 + j)] * bo);
            }
            m[nt][j] = mn;
          }
        }
      }
      named_barrier(1, nwc * 32);
    }
    if (kg == 0) {
      float* dstp = p.partials + ((size_t)(blockIdx.x + seg) * R) * kPartialStride;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tile = tg * NT + nt;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float lt = warp_sum_g(l[nt][j]);
          const float ot = warp_sum_g(ov[nt][j]);
          const int row = 8 * tile + 2 * t + j;
          if (row >= R) continue;
          float* dst = dstp + (size_t)row * kPartialStride;
          if (g == 0) {
            dst[0] = m[nt][j];
            dst[1] = lt;
          }
          const float vs = FMT == 0 ? 1.0f : p.v_scale;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int dlo = out_dim<FMT>(i, g), dhi = out_dim<FMT>(i, g + 8);
            if (FMT == 0) {  // V entered as unpack8_v values: dims of class 2 (i & 1) and 2 (i & 1) + 1
              dst[2 + dlo] = fmaf(acc[nt][i][j], v_unscale(2 * (i & 1)), ot);
              dst[2 + dhi] = fmaf(acc[nt][i][2 + j], v_unscale(2 * (i & 1) + 1), ot);
            } else {
              dst[2 + dlo] = (acc[nt][i][j] + ot) * vs;
              dst[2 + dhi] = (acc[nt][i][2 + j] + ot) * vs;
            }
          }
        }
      }
    }
    seg_start = seg_end;
  }

}

// ------------------------------------------------------------ many query rows: tcgen05 kernel
// Verify blocks put S x G query rows (up to 48) on every KV head; both products then are small
// dense contractions per 128 tokens, run here as tcgen05.mma with the accumulators in tensor
// memory and the converted K and V codes there as well (A operands read from tensor memory), so
// that shared memory carries only the page copies, the query tile Q', the probabilities P and
// the per-token scales. Work split and partials are those of attn_kernel (stream-K over pages,
// combine_kernel after).
//
// Units: up to two pages (128 tokens) of one segment. Within each 16-token group the tokens
// take the order sigma(k) = 2 (k >> 2 & 3) + 8 (k >> 1 & 1) + (k & 1) (k = 0..15) along the
// contraction of PV, so that the V fragments of ldmatrix.trans + unpack8_v store as
// tcgen05.st.16x256b blocks; QK^T uses the same order for its M index (tensor-memory lane k
// holds token sigma(k)), and so does the row order of P.
//
//   warps 0-3   converters: warp q owns tensor-memory lanes 32q..32q+31. Per unit: the K codes of
//               unit tokens sigma(32q + lane) -> exact f16 subnormals (unpack8_sub) -> A_K
//               (tcgen05.st.32x32b), their scales and offsets -> shared memory; the V codes of
//               dims 32q + 4g + 2e + h of both pages -> ldmatrix.trans -> unpack8_v (exact
//               centred f16 subnormals) -> A_V lanes 32q + 16e + 8h + g (tcgen05.st.16x256b).
//   warps 4-11  softmax: warp 4 + 4 grp + q owns lanes 32q..32q+31 (the unit's tokens) and row
//               half grp (rows grp*H .. grp*H + H - 1, H = NR / 2): its token's scores from S,
//               the online softmax (lazy base as attn_kernel, decided per row half), P = p s_V
//               in f16 into shared memory (MN-major, 128-byte swizzle); at a segment end the
//               row sums, the next segment's Q' rows and the partial rows from O.
//   warp 12     producer (produce_pages into kTcStages stages).
//   warp 13     tensor-memory allocation and the QK issue: S[u&1] = A_K Q'^T (M = 128 tokens,
//               N = NR rounded up to 16, K = 128 dims, Q' K-major).
//   warp 14     the PV issue: O += A_V P (M = 128 dims, N, K = tokens, P MN-major). One issuing
//               thread for both products would be the slowest part of a unit: it shares its
//               scheduler with converter and softmax warps, and a unit takes 16 MMAs.
//   warp 15     idle (completes the warpgroup of 12-14 for the register split).
// Conversion of unit u + 1 runs on the converters while the softmax warps work on unit u.
// Tensor memory: A_K[2] cols 0..127, A_V[3] 128..319, S[2] 320..447, O 448..511 (512 allocated).
constexpr int kTcStages = 8;
// Calls with more query rows per KV head than this take the tcgen05 kernel; up to 16 rows the
// split kernel's mma.sync tiles finish first (measured: 16 rows 179 us there, 222 us here, on
// 64 x 16,384 tokens; 20 rows 249 us there, 235 us here).
constexpr int kTcMinRows = 16;
constexpr int kTcWarps = 16;  // warp 15 only completes the last warpgroup (setmaxnreg is per warpgroup)
// registers per thread of the converters (warps 0-3), the softmax warps (4-11) and the producer /
// issuer warpgroup (12-15), set by setmaxnreg from the launch's 128
constexpr int kTcRegConv = 96, kTcRegSoftmax = 168, kTcRegAux = 64;
static_assert(128 * kTcRegConv + 256 * kTcRegSoftmax + 128 * kTcRegAux <= kTcWarps * 32 * 128,
              "register shares above the launch's allocation");
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcMaxRows = 48;
constexpr uint32_t kColAK = 0, kColAV = 128, kColS = 320, kColO = 448;
constexpr int kTcHalf = kTcMaxRows * 128;  // bytes of one 64-dim half of Q'
constexpr int kTcBars = 32;                // mbarriers of the kernel (see its list)

struct TcLayout {  // offsets from the 1024-byte aligned start of dynamic shared memory
  size_t stages, qt, pt, meta, bars, valid, flags, taddr, uinfo, rowc, rowst, ovrow, red, rowm, rcx, rcy, ralpha, rdelta,
      pre, total;
  __host__ __device__ explicit TcLayout(int B) {
    stages = 0;
    qt = kTcStages * (size_t)kStage4;  // 69632 = 68 * 1024
    pt = qt + 2 * kTcHalf;             // + 12288
    meta = pt + 3 * 128 * 128;         // P[3]: 128 token rows of 128 bytes
    bars = meta + 3 * 128 * 16;        // per-token (k scale, k offset, v scale, v term) of 3 units
    valid = bars + 8 * kTcBars;
    flags = valid + 4 * kTcStages;
    taddr = flags + 16;
    uinfo = align_up(taddr + 16, 16);
    rowc = uinfo + 3 * 16;
    rowst = rowc + 16 * kTcMaxRows;
    ovrow = rowst + 4 * kTcMaxRows;
    red = ovrow + 4 * kTcMaxRows;
    rowm = red + 4 * 2 * 4 * kTcMaxRows;
    rcx = rowm + 4 * 4 * kTcMaxRows;
    rcy = rcx + 4 * kTcMaxRows;
    ralpha = rcy + 4 * kTcMaxRows;
    rdelta = ralpha + 4 * kTcMaxRows;
    pre = rdelta + 4 * kTcMaxRows;
    total = align_up(pre + 4 * (size_t)(B + 1), 16);
  }
};

// The CTA's pages [p0, p1) as units of up to two pages of one segment, in order.
struct TcUnits {
  const AttnParams& p;
  const int* pre;
  long long p0, p1, k, seg_start, seg_end, ustart;
  int b, h, lp0, np, segi, npg;
  bool first, last;
  __device__ TcUnits(const AttnParams& p_, const int* pre_, long long a, long long e)
      : p(p_), pre(pre_), p0(a), p1(e), k(a), seg_start(0), seg_end(-1), ustart(0), b(0), h(0), lp0(0), np(1),
        segi(-1), npg(0), first(false), last(false) {}
  __device__ bool next() {
    if (k >= p1) return false;
    if (k >= seg_end) {
      decode_page(pre, p.B, p.Hkv, k, b, h, lp0, np);
      seg_start = k;
      seg_end = min(p1, k + (np - lp0));
      ++segi;
      first = true;
    } else {
      first = false;
    }
    ustart = k;
    npg = (int)min(2LL, seg_end - k);
    k += npg;
    last = k >= seg_end;
    return true;
  }
  __device__ int lp() const { return lp0 + (int)(ustart - seg_start); }  // local page of the unit's first page
  __device__ int kidx() const { return (int)(ustart - p0); }              // CTA page index of that page
};

// Token of unit lane k (0..127): 16 (k >> 4) + sigma(k & 15).
__device__ __forceinline__ int tc_token(int k) {
  return (k & ~15) + 2 * ((k >> 2) & 3) + 8 * ((k >> 1) & 1) + (k & 1);
}

// Byte offset of K-index kd (0..127) of row r in Q' (K-major, two 64-index halves of rows of 128
// bytes, 8-row groups, 16-byte chunk c of row r at c ^ (r & 7)).
__device__ __forceinline__ int tc_q_offset(int r, int kd) {
  return (kd >> 6) * kTcHalf + r * 128 + 16 * (((kd & 63) >> 3) ^ (r & 7)) + 2 * (kd & 7);
}

// NR: softmax rows of the CTA (R rounded up to 8, at most 48); the MMAs take N = NR rounded up
// to 16 (P columns beyond NR are never written: their D columns are not read).
template <int NR>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const AttnParams p) {
  constexpr int H = NR / 2;  // rows of one softmax group (a multiple of 4)
  constexpr int NM = (NR + 15) & ~15;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const TcLayout L(p.B);
  uint8_t* stages = smem + L.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* full = bars;            // [8] page copied
  uint64_t* empty = bars + 8;       // [8] page read (the 4 converters)
  uint64_t* cready = bars + 16;     // [3] A_K[u & 1], A_V[u % 3] and the scales of unit u written
  uint64_t* sfull = bars + 19;      // [2] QK(u) done
  uint64_t* pready = bars + 21;     // [3] P[u % 3] of unit u written (so S[u & 1] has been read)
  uint64_t* vfree = bars + 24;      // [3] PV(u) done: A_V, P and scales of u % 3 free
  uint64_t* qready = bars + 27;     // Q' of a segment written (both groups)
  uint64_t* ofull = bars + 28;      // a segment's last PV done
  uint64_t* ofree = bars + 29;      // O of a segment read (both groups)
  uint64_t* fin = bars + 30;        // [2] final MMA completion of the QK / PV issuer
  static_assert(31 < kTcBars, "mbarrier list larger than its shared-memory region");
  volatile int* valid = reinterpret_cast<volatile int*>(smem + L.valid);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + L.flags);
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(smem + L.taddr);
  float4* tmeta = reinterpret_cast<float4*>(smem + L.meta);  // [3][128 unit lanes]
  float4* rowc = reinterpret_cast<float4*>(smem + L.rowc);    // (qs * scale, -muse, threshold, last position)
  float* rowst = reinterpret_cast<float*>(smem + L.rowst);    // running maximum m (log2 units)
  float* ovrow = reinterpret_cast<float*>(smem + L.ovrow);
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* rowm = reinterpret_cast<float*>(smem + L.rowm);
  // descriptor of unit u in slot u % 3, written by converter warp 0 before its cready(u) arrival:
  // (sequence | head << 16, local page of its first page, pages | first << 2 | last << 3 |
  // final << 4, CTA page index after it). The slot is rewritten only after PV(u) completed.
  int4* uinfo = reinterpret_cast<int4*>(smem + L.uinfo);
  float* rcx = reinterpret_cast<float*>(smem + L.rcx);        // rowc x and y by row, for 16-byte loads
  float* rcy = reinterpret_cast<float*>(smem + L.rcy);
  float* ralpha = reinterpret_cast<float*>(smem + L.ralpha);  // a base move: factor on a row's sums and O
  float* rdelta = reinterpret_cast<float*>(smem + L.rdelta);  // and shift of its scores
  int* pre = reinterpret_cast<int*>(smem + L.pre);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr uint32_t kFinBar = 1;
  constexpr int kGrp = 128, kFinThreads = 14 * 32;

  // The setup (page prefix from the context lengths, barriers, Q' padding, tensor memory) runs
  // while the previous grid, the call's prologue/append kernel, finishes; see attn_kernel. Every
  // grid before it has completed, so no earlier kernel of the stream still holds tensor memory.
  build_prefix(p, 0, pre, flags);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&sfull[b], 1);
    for (int b = 0; b < 3; ++b) {
      mbar_init(&cready[b], 4);
      mbar_init(&pready[b], 8);
      mbar_init(&vfree[b], 1);
    }
    mbar_init(qready, 2);
    mbar_init(ofull, 1);
    mbar_init(ofree, 2);
    mbar_init(&fin[0], 1);
    mbar_init(&fin[1], 1);
  }
  // Q' rows beyond R stay zero
  for (int i = threadIdx.x; i < 2 * kTcHalf / 16; i += kTcThreads)
    reinterpret_cast<uint4*>(smem + L.qt)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_barrier_init();
  fence_proxy_async_shared();
  if (warp == 13) tmem_alloc_512(taddr_s);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *taddr_s;
  griddep_wait();
  griddep_launch_dependents();

  if (blockIdx.x == 0 && threadIdx.x == 0 && flags[1]) set_err(p.dev_err, KVQ_DEVERR_POS);
  const long long P = (long long)p.Hkv * pre[p.B];
  const int n_eff = (int)min((long long)p.n_cta, P);
  const bool active = (int)blockIdx.x < n_eff;
  const long long p0 = active ? (long long)blockIdx.x * P / n_eff : 0;
  const long long p1 = active ? (long long)(blockIdx.x + 1) * P / n_eff : 0;
  const int R = p.R, G = p.G;

  // Registers per thread by warpgroup: the softmax warps hold a score and two running sums per
  // row; the producer and issuer threads need few. The shares add up to at most the launch's
  // 128 per thread (setmaxnreg.inc waits for registers released by .dec).
  // Each role's code is entered only after its warpgroup's setmaxnreg and ends in a return.
  if (warp >= 12) {
  reg_dealloc<kTcRegAux>();
  if (warp == 15) return;

  // ------------------------------------------------------------ producer
  if (warp == 12) {
    if (active) produce_pages<0>(p, pre, stages, full, empty, valid, flags, kTcStages, p0, p1, lane);
    return;
  }

  // ------------------------------------------------------------ MMA issue
  // Two issuing threads, each on its own scheduler: warp 13 issues QK, warp 14 PV. A commit
  // tracks only its own thread's MMAs; the two write disjoint tensor memory (S, O) and read
  // operands whose reuse each side orders on its own barriers. PV(u) reads A_V[u % 3]: it was
  // written before cready(u), which the softmax warps waited for before they arrived on pready(u).
  {  // warps 13 and 14
    if (lane == 0 && active) {
      bool ok = true;
      int b3 = 0;       // unit % 3
      uint32_t ph3 = 0;  // (unit / 3) & 1
      int segi = -1;    // segment of the unit
      if (warp == 13) {
        const uint32_t idesc = umma_idesc_f16(NM, false, false);
        const uint64_t dq = umma_sdesc(smem_addr(smem + L.qt), 16, 1024);
        int pb3 = 0;       // (unit - 2) % 3, from unit 2 on
        uint32_t pph3 = 0;  // ((unit - 2) / 3) & 1
        for (int v = 0;; ++v) {
          const int b = v & 1;
          ok = mbar_wait_bounded(&cready[b3], ph3);
          if (!ok) break;
          const int uz = uinfo[b3].z;
          if (uz & 4) ++segi;
          // S[b] was read before P of unit v - 2 was written
          ok = v < 2 || mbar_wait_bounded(&pready[pb3], pph3);
          ok = ok && (!(uz & 4) || mbar_wait_bounded(qready, (uint32_t)segi & 1u));
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem + kColS + 64 * b, a0 = tmem + kColAK + 64 * b;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // k-steps of 16 dims: 32 bytes within a 64-dim half
            umma_f16_ts(d, a0 + 8 * kk, dq + (uint64_t)(((kk >> 2) * kTcHalf + (kk & 3) * 32) >> 4), idesc, kk > 0);
          umma_commit(&sfull[b]);
          if (++b3 == 3) { b3 = 0; ph3 ^= 1u; }
          if (v >= 2 && ++pb3 == 3) { pb3 = 0; pph3 ^= 1u; }
          if (uz & 16) break;  // the CTA's last unit
        }
      } else {
        const uint32_t idesc = umma_idesc_f16(NM, false, true);
        const uint64_t dp = umma_sdesc(smem_addr(smem + L.pt), 16384, 1024);
        for (;;) {
          ok = mbar_wait_bounded(&pready[b3], ph3);
          if (!ok) break;
          const int uz = uinfo[b3].z;  // P(u) written implies cready(u) was seen
          if (uz & 4) ++segi;
          ok = !(uz & 4) || segi == 0 || mbar_wait_bounded(ofree, (uint32_t)(segi - 1) & 1u);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = tmem + kColAV + 64 * b3;
          const uint64_t d0 = dp + (uint64_t)(b3 * (16384 >> 4));
          const uint32_t acc0 = (uz & 4) ? 0u : 1u;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // k-steps of 16 tokens: 2048 bytes of P each
            umma_f16_ts(tmem + kColO, a0 + 8 * kk, d0 + (uint64_t)(kk * (2048 >> 4)), idesc, kk > 0 ? 1u : acc0);
          if ((uz & 3) == 2) {
#pragma unroll
            for (int kk = 4; kk < 8; ++kk)
              umma_f16_ts(tmem + kColO, a0 + 8 * kk, d0 + (uint64_t)(kk * (2048 >> 4)), idesc, 1u);
          }
          umma_commit(&vfree[b3]);
          if (uz & 8) umma_commit(ofull);
          if (++b3 == 3) { b3 = 0; ph3 ^= 1u; }
          if (uz & 16) break;  // the CTA's last unit
        }
      }
      if (!ok) {
        set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
        flags[0] = 1;
      }
      uint64_t* done = warp == 13 ? fin : fin + 1;
      umma_commit(done);  // every MMA this thread issued has completed once this arrives
      if (!mbar_wait_bounded(done, 0)) set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
    }
    __syncwarp();
    tc_fence_before();
    named_barrier(kFinBar, kFinThreads);
    tc_fence_after();
    if (warp == 13) tmem_dealloc_512(tmem);
    return;
  }
  }  // warps 12-15

  // ------------------------------------------------------------ converters
  if (warp < 4) {
    reg_dealloc<kTcRegConv>();
    const int q = warp;
    const int kl = 32 * q + lane;              // unit lane of this thread's token
    const int tok = tc_token(kl);              // token of the unit (0..127)
    const int jj = tok >> 6, slot = tok & 63;  // its page (warp-uniform) and slot
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    TcUnits Uc(p, pre, p0, p1);
    bool ok = true;
    int bv = 0;           // u % 3
    uint32_t fph = 1;     // ((u - 3) / 3) & 1 for vfree, from u = 3 on (flipped before use)
    for (int u = 0; active && ok && Uc.next(); ++u) {
      const int bk = u & 1;
      if (u >= 3 && bv == 0) fph ^= 1u;
      // A_V, P and scales of u % 3 were last used by PV(u - 3); A_K[u & 1] by QK(u - 2). Every
      // barrier of the unit is tested at once; only an incomplete one is waited for in turn.
      const int kp0 = Uc.kidx(), npg = Uc.npg;
      const int s0 = kp0 % kTcStages, s1 = (kp0 + 1) % kTcStages;
      const uint32_t f0 = (uint32_t)(kp0 / kTcStages) & 1u, f1 = (uint32_t)((kp0 + 1) / kTcStages) & 1u;
      const uint32_t sph = (uint32_t)((u - 2) >> 1) & 1u;
      bool ready = mbar_test(&full[s0], f0);
      if (npg == 2) ready &= mbar_test(&full[s1], f1);
      if (u >= 3) ready &= mbar_test(&vfree[bv], fph);
      if (u >= 2) ready &= mbar_test(&sfull[bk], sph);
      if (!__all_sync(0xffffffffu, ready)) {
        bool w = u < 3 || mbar_wait_bounded(&vfree[bv], fph);
        w = w && (u < 2 || mbar_wait_bounded(&sfull[bk], sph));
        w = w && mbar_wait_bounded(&full[s0], f0);
        w = w && (npg < 2 || mbar_wait_bounded(&full[s1], f1));
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
      }
      // ---- K: this thread's token (page jj) -> A_K[u & 1], its scales -> shared memory
      float4 mt = make_float4(0.f, 0.f, -1.f, 0.f);  // v scale -1: no token
      if (jj < npg) {
        const int s = jj ? s1 : s0;
        const uint8_t* st = stages + (size_t)s * kStage4;
        const int sw = k_chunk_swz(slot);
        const uint8_t* rec = st + slot * kRec4;
        const bool vld = valid[s] != 0;
        const uint32_t mk = reinterpret_cast<const uint32_t*>(st + 2 * kPage * kRec4)[slot];
        const uint32_t mv = reinterpret_cast<const uint32_t*>(st + 2 * kPage * kRec4)[kPage + slot];
        // chunk c (words 4c..4c+3) -> columns 16c .. 16c + 15, each chunk's load issued one chunk
        // ahead; fully unrolled (measured on 64 x 16,384 tokens: a rolled loop or one unrolled by
        // two, kept for the instruction cache in earlier forms of the kernel, now costs 8-16 us)
        uint4 kc = *reinterpret_cast<const uint4*>(rec + 16 * sw);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 kn = *reinterpret_cast<const uint4*>(rec + 16 * (((c + 1) & 3) ^ sw));
          const uint32_t wd[4] = {kc.x, kc.y, kc.z, kc.w};
          uint32_t w16[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t h4[4];
            unpack8_sub(wd[i], h4);
#pragma unroll
            for (int j = 0; j < 4; ++j) w16[4 * i + j] = h4[j];
          }
          tmem_st16u(tmem + lane_base + kColAK + 64 * bk + 16 * c, w16);
          kc = kn;
        }
        if (vld) {
          const float sv = h2f_lo(mv);
          mt = make_float4(h2f_lo(mk) * p.score_scale * 16777216.0f, h2f_hi(mk), sv, fmaf(7.5f, sv, h2f_hi(mv)));
        }
      }
      tmeta[bv * 128 + kl] = mt;
      // ---- V codes of dims 32q .. 32q + 31 of both pages: every ldmatrix before any conversion
      uint32_t rr[2][2][4];  // [page][half of the page]
#pragma unroll
      for (int pg = 0; pg < 2; ++pg) {
        if (pg < npg) {
          const uint8_t* Vs = stages + (size_t)(pg ? s1 : s0) * kStage4 + kPage * kRec4;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int t8 = 32 * hf + 8 * (lane >> 3) + (lane & 7);
            ldsm_x4_trans(rr[pg][hf], smem_addr(Vs + t8 * kRec4 + 16 * (q ^ ((t8 >> 1) & 3))));
          }
        }
      }
      __syncwarp();
      mbar_arrive_if(&empty[s0], lane == 0);  // both pages read (K above, V into registers)
      if (npg == 2) mbar_arrive_if(&empty[s1], lane == 0);
#pragma unroll
      for (int pg = 0; pg < 2; ++pg) {
        if (pg < npg) {
          uint32_t ra[16], rb[16];  // dims of class 2e + h at lanes 32q + 16e + 8h + g, e = 0 / 1
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
            for (int gq = 0; gq < 2; ++gq) {
              uint32_t h0[4], h1[4];
              unpack8_v(rr[pg][hf][2 * gq], h0);      // tokens 16 gq + 2t, +1 of this half
              unpack8_v(rr[pg][hf][2 * gq + 1], h1);  // tokens 16 gq + 8 + 2t, +1
              const int j = 2 * hf + gq;              // 16-token group of the page
              ra[4 * j] = h0[0];
              ra[4 * j + 1] = h1[0];
              ra[4 * j + 2] = h0[1];
              ra[4 * j + 3] = h1[1];
              rb[4 * j] = h0[2];
              rb[4 * j + 1] = h1[2];
              rb[4 * j + 2] = h0[3];
              rb[4 * j + 3] = h1[3];
            }
          }
          const uint32_t col = tmem + kColAV + 64 * bv + 32 * pg;
          tmem_st_16x256b_x4(col + lane_base, ra);
          tmem_st_16x256b_x4(col + ((uint32_t)(32 * q + 16) << 16), rb);
        }
      }
      if (q == 0 && lane == 0)
        uinfo[bv] = make_int4(Uc.b | (Uc.h << 16), Uc.lp(),
                              npg | (Uc.first ? 4 : 0) | (Uc.last ? 8 : 0) | (Uc.k >= p1 ? 16 : 0), (int)(Uc.k - p0));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      mbar_arrive_if(&cready[bv], lane == 0);
      if (++bv == 3) bv = 0;
    }
    if (!ok) {
      if (lane == 0) set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
      flags[0] = 1;
    }
    tc_fence_before();
    named_barrier(kFinBar, kFinThreads);
    return;
  }

  // ------------------------------------------------------------ softmax warps
  reg_alloc<kTcRegSoftmax>();
  const int q = warp & 3, grp = (warp - 4) >> 2;  // lane quarter, row half
  const uint32_t kGrpBar = 2 + grp;               // named barrier of the row half
  const int kl = 32 * q + lane;                   // unit lane: row of S and of P
  const int tok = tc_token(kl);                   // token of the unit (0..127)
  const int jj = tok >> 6, slot = tok & 63;       // page of the unit (warp-uniform) and slot
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  const int gt = threadIdx.x - 128 - 128 * grp;   // 0..127 within the row half
  const int r0 = grp * H;                         // first row of the half
  // running sums of p and of p * (v term) of this thread's tokens; pair i holds rows 2i, 2i + 1
  uint64_t l2[H / 2], ov2[H / 2];
#pragma unroll
  for (int i = 0; i < H / 2; ++i) l2[i] = ov2[i] = 0ull;  // (0.0f, 0.0f)

  // Q' rows and row constants of this half for segment (bq, hq): K-index kd of a row holds dim
  // 8w + j + 4e (kd = 8w + 2j + e, the order of unpack8_sub), divided by 16 for odd j. Row
  // constants: (sum q~ * scale, -base (0 while the base is -inf; -inf on padding rows, whose
  // scores then are -inf), threshold of the lazy base (+inf on padding rows), last visible
  // position of the row's query).
  auto load_segment = [&](int bq, int hq) -> int {
    bool bad = false;
    const int cb = eff_ctx(p, bq, bad, 0);
#pragma unroll 1
    for (int e = gt; e < H * 16; e += kGrp) {
      const int r = r0 + (e >> 4), w = e & 15;
      float part = 0.0f;
      uint32_t hq4[4];
      if (r < R) {
        const float* qrow = p.q_rot + (((size_t)bq * p.S + r / G) * p.Hq + hq * G + r % G) * kD + 8 * w;
        const float4 a = reinterpret_cast<const float4*>(qrow)[0], c4 = reinterpret_cast<const float4*>(qrow)[1];
        const float qv[8] = {a.x, a.y, a.z, a.w, c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) part += qv[i];
        hq4[0] = pack_f16x2(qv[0], qv[4]);
        hq4[1] = pack_f16x2(qv[1] * 0.0625f, qv[5] * 0.0625f);
        hq4[2] = pack_f16x2(qv[2], qv[6]);
        hq4[3] = pack_f16x2(qv[3] * 0.0625f, qv[7] * 0.0625f);
      } else {
        hq4[0] = hq4[1] = hq4[2] = hq4[3] = 0u;
      }
      *reinterpret_cast<uint4*>(smem + L.qt + tc_q_offset(r, 8 * w)) = make_uint4(hq4[0], hq4[1], hq4[2], hq4[3]);
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (w == 0) {
        const float4 c = r < R ? make_float4(part * p.score_scale, 0.0f, -INFINITY, (float)(cb + r / G))
                               : make_float4(0.0f, -INFINITY, INFINITY, -1.0f);
        rowc[r] = c;
        rcx[r] = c.x;
        rcy[r] = c.y;
        rowst[r] = -INFINITY;
      }
    }
    fence_proxy_async_shared();
    return cb;
  };

  // units come from the descriptors in uinfo; the next segment's Q' is loaded at a segment end
  bool more = active;
  bool err = false;
  int ctx_next = 0;  // effective context length of the next segment
  if (more) {
    int b0, h0, lpf, npf;
    decode_page(pre, p.B, p.Hkv, p0, b0, h0, lpf, npf);
    ctx_next = load_segment(b0, h0);
  }
  err = named_barrier_or(kGrpBar, kGrp, false);
  if (more && gt == 0) mbar_arrive(qready);
  int ctxb = 0, segi = -1;
  // smallest lazy-base threshold over the half's rows (-inf until every row has a base)
  float thr_grp = -INFINITY;
  // segments; within one, its units (the hot loop), then the segment end after it
  int v = 0;
  while (more && !err) {
    int4 ui;  // the unit's descriptor; after the unit loop, the segment's last unit's
    for (;;) {
      const int b = v & 1, bv = v % 3;
      // waits are made warp-uniform: the tensor-memory loads after them are warp-collective
      bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&sfull[b], (uint32_t)(v >> 1) & 1u) &&
                                            mbar_wait_bounded(&cready[bv], (uint32_t)(v / 3) & 1u));
      ui = uinfo[bv];
      const int ulp = ui.y, unpg = ui.z & 3;
      const bool ufirst = (ui.z & 4) != 0, ulast = (ui.z & 8) != 0;
      if (ufirst) {
        ctxb = ctx_next;
        ++segi;
      }
      float d[H];
      if (ok) {
        tc_fence_after();
  #pragma unroll
        for (int c = 0; c < H / 4; ++c) {
          float t4[4];
          tmem_ld4(tmem + lane_base + kColS + 64 * b + r0 + 4 * c, t4);
  #pragma unroll
          for (int i = 0; i < 4; ++i) d[4 * c + i] = t4[i];
        }
        tmem_wait_ld();
      }
      tc_fence_before();
      const float4 mt = tmeta[bv * 128 + kl];  // (k scale * score scale * 2^24, k offset, v scale, v term)

      // ---- scores of this token relative to each row's base; branch-free over the rows (padding
      // rows carry a -inf base); the causal limits apply only on a unit that reaches past the context
      const bool tvalid = ok && mt.z >= 0.0f;
      const bool unit_mask = (ulp + unpg) * kPage - 1 > ctxb;
      float mx = -INFINITY;
      if (!tvalid) {
  #pragma unroll
        for (int i = 0; i < H; ++i) d[i] = -INFINITY;
      } else if (!unit_mask) {
        // d mt.x + (mt.y c.x + c.y), four rows at a time in fp32 pairs
        const uint64_t mtx2 = f2(mt.x, mt.x), mty2 = f2(mt.y, mt.y);
  #pragma unroll
        for (int c = 0; c < H / 4; ++c) {
          const float4 cx = reinterpret_cast<const float4*>(rcx + r0)[c];
          const float4 cy = reinterpret_cast<const float4*>(rcy + r0)[c];
          const uint64_t s01 = fma_f2(f2(d[4 * c], d[4 * c + 1]), mtx2, fma_f2(mty2, f2(cx.x, cx.y), f2(cy.x, cy.y)));
          const uint64_t s23 = fma_f2(f2(d[4 * c + 2], d[4 * c + 3]), mtx2, fma_f2(mty2, f2(cx.z, cx.w), f2(cy.z, cy.w)));
          d[4 * c] = f2lo(s01);
          d[4 * c + 1] = f2hi(s01);
          d[4 * c + 2] = f2lo(s23);
          d[4 * c + 3] = f2hi(s23);
          mx = fmax3(mx, d[4 * c], d[4 * c + 1]);
          mx = fmax3(mx, d[4 * c + 2], d[4 * c + 3]);
        }
      } else {
        const float fpos = (float)((ulp + jj) * kPage + slot);
  #pragma unroll
        for (int i = 0; i < H; ++i) {
          const float4 c = rowc[r0 + i];
          const float sc = fmaf(d[i], mt.x, fmaf(mt.y, c.x, c.y));
          d[i] = fpos <= c.w ? sc : -INFINITY;
          mx = fmaxf(mx, d[i]);
        }
      }
      const bool need = mx > (mt.z >= 255.0f ? fminf(thr_grp, 0.0f) : thr_grp);  // large V scale: any excess
      if (__builtin_expect(named_barrier_or(kGrpBar, kGrp, need || !ok), 0)) {
        err = named_barrier_or(kGrpBar, kGrp, !ok);
        if (err) break;
        // ---- rare: move the base of the rows whose maximum passed it (row maxima over the 128 tokens)
  #pragma unroll
        for (int i = 0; i < H; ++i) {
          const float m1 = warp_max_all(d[i]);
          if (lane == 0) rowm[q * kTcMaxRows + r0 + i] = m1;
        }
        named_barrier(kGrpBar, kGrp);
        // one thread per row: the new base (published), the factor alpha on the row's sums and O
        // and the shift of this unit's scores to the new base (1 and 0 where the base stays)
        bool changed = false;
        if (gt < H) {
          const int r = r0 + gt;
          float alpha = 1.0f, delta = 0.0f;
          if (r < R) {
            const float mt4 = fmaxf(fmaxf(rowm[r], rowm[kTcMaxRows + r]), fmaxf(rowm[2 * kTcMaxRows + r], rowm[3 * kTcMaxRows + r]));
            const float4 c = rowc[r];
            const float mold = rowst[r], muse = -c.y;
            const float mnew = fmaxf(mold, muse + mt4);
            if (mnew != mold) {
              const float mu2 = mnew == -INFINITY ? 0.0f : mnew;
              alpha = fast_exp2(mold - mu2);
              delta = muse - mu2;
              changed = true;
              const float nb = mnew == -INFINITY ? 0.0f : -mnew;
              rowst[r] = mnew;
              rowc[r] = make_float4(c.x, nb, mnew == -INFINITY ? -INFINITY : 8.0f, c.w);
              rcy[r] = nb;
            }
          }
          ralpha[r] = alpha;
          rdelta[r] = delta;
        }
        if (named_barrier_or(kGrpBar, kGrp, changed)) {
  #pragma unroll
          for (int i = 0; i < H / 2; ++i) {
            const uint64_t a2 = f2(ralpha[r0 + 2 * i], ralpha[r0 + 2 * i + 1]);
            l2[i] = mul_f2(l2[i], a2);
            ov2[i] = mul_f2(ov2[i], a2);
          }
  #pragma unroll
          for (int i = 0; i < H; ++i) d[i] += rdelta[r0 + i];
          // O (this thread's lane, the half's rows) -- not on a segment's first unit: O starts from
          // zero there. PV(v - 1) must have completed.
          if (!ufirst) {
            const bool okp = __all_sync(0xffffffffu, mbar_wait_bounded(&vfree[(v - 1) % 3], (uint32_t)((v - 1) / 3) & 1u));
            if (okp) {
              tc_fence_after();
  #pragma unroll
              for (int c = 0; c < H / 4; ++c) {
                float t4[4];
                tmem_ld4(tmem + lane_base + kColO + r0 + 4 * c, t4);
                tmem_wait_ld();
  #pragma unroll
                for (int i = 0; i < 4; ++i) t4[i] *= ralpha[r0 + 4 * c + i];
                tmem_st4(tmem + lane_base + kColO + r0 + 4 * c, t4);
              }
              tmem_wait_st();
            }
            tc_fence_before();
            err = named_barrier_or(kGrpBar, kGrp, !okp);
            if (err) break;
          }
        }
        thr_grp = INFINITY;
  #pragma unroll
        for (int i = 0; i < H; ++i)
          if (r0 + i < R) thr_grp = fminf(thr_grp, rowc[r0 + i].z);
      }

      // ---- P s_V in f16 (row kl of P[v % 3], MN-major: query row r at byte 2 (r & 7) of chunk r >> 3)
      uint32_t pk[H / 2];
      const uint64_t mtz2 = f2(mt.z, mt.z), mtw2 = f2(mt.w, mt.w);
  #pragma unroll
      for (int i = 0; i < H / 2; ++i) {
        const uint64_t pp = f2(fast_exp2(d[2 * i]), fast_exp2(d[2 * i + 1]));
        l2[i] = add_f2(l2[i], pp);
        ov2[i] = fma_f2(pp, mtw2, ov2[i]);
        const uint64_t ps = mul_f2(pp, mtz2);
        pk[i] = pack_f16x2_sat(f2lo(ps), f2hi(ps));
      }
      // P[v % 3] was read by PV(v - 3), complete since the converters waited for it before
      // writing this unit's codes (cready above)
      {
        uint8_t* prow = smem + L.pt + bv * 16384 + kl * 128;
  #pragma unroll
        for (int m = 0; m < H / 4; ++m) {  // rows r0 + 4m .. + 3 (8 bytes)
          const int r = r0 + 4 * m;
          *reinterpret_cast<uint2*>(prow + 16 * ((r >> 3) ^ (kl & 7)) + 2 * (r & 7)) = make_uint2(pk[2 * m], pk[2 * m + 1]);
        }
        fence_proxy_async_shared();
      }
      __syncwarp();
      mbar_arrive_if(&pready[bv], lane == 0);
      ++v;
      if (ulast) break;
    }
    if (err) break;

    {
      // ---- segment end: token sums per row, the next segment's Q', then O -> CTA partial
      const int seg = (ui.x & 0xFFFF) * p.Hkv + (ui.x >> 16);
#pragma unroll
      for (int i = 0; i < H; ++i) {
        float lt = (i & 1) ? f2hi(l2[i / 2]) : f2lo(l2[i / 2]);
        float ot = (i & 1) ? f2hi(ov2[i / 2]) : f2lo(ov2[i / 2]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          lt += __shfl_xor_sync(0xffffffffu, lt, o);
          ot += __shfl_xor_sync(0xffffffffu, ot, o);
        }
        if (lane == 0) {
          red[(q * kTcMaxRows + r0 + i) * 2] = lt;
          red[(q * kTcMaxRows + r0 + i) * 2 + 1] = ot;
        }
      }
#pragma unroll
      for (int i = 0; i < H / 2; ++i) l2[i] = ov2[i] = 0ull;
      named_barrier(kGrpBar, kGrp);
      if (gt < H && r0 + gt < R) {
        const int r = r0 + gt;
        float lt = 0.0f, ot = 0.0f;
        for (int qq = 0; qq < 4; ++qq) {
          lt += red[(qq * kTcMaxRows + r) * 2];
          ot += red[(qq * kTcMaxRows + r) * 2 + 1];
        }
        float* dst = p.partials + ((size_t)(blockIdx.x + seg) * R + r) * kPartialStride;
        dst[0] = rowst[r];
        dst[1] = lt;
        ovrow[r] = ot;
      }
      named_barrier(kGrpBar, kGrp);
      const bool nmore = (ui.z & 16) == 0;
      if (nmore) {
        int nb, nh, nlp, nnp;
        decode_page(pre, p.B, p.Hkv, p0 + ui.w, nb, nh, nlp, nnp);
        ctx_next = load_segment(nb, nh);
      }
      named_barrier(kGrpBar, kGrp);
      if (nmore && gt == 0) mbar_arrive(qready);
      thr_grp = -INFINITY;
      // O of the finished segment: lane kl holds dim 32q + 4g + 2e + h for kl = 32q + 16e + 8h + g
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(ofull, (uint32_t)segi & 1u));
      if (ok) {
        tc_fence_after();
        float o[H];
#pragma unroll
        for (int c = 0; c < H / 4; ++c) {
          float t4[4];
          tmem_ld4(tmem + lane_base + kColO + r0 + 4 * c, t4);
#pragma unroll
          for (int i = 0; i < 4; ++i) o[4 * c + i] = t4[i];
        }
        tmem_wait_ld();
        const int e = (lane >> 4) & 1, hh = (lane >> 3) & 1, g = lane & 7;
        const int dim = 32 * q + 4 * g + 2 * e + hh;
        const float us = v_unscale(dim & 3);
#pragma unroll
        for (int i = 0; i < H; ++i)
          if (r0 + i < R)
            p.partials[((size_t)(blockIdx.x + seg) * R + r0 + i) * kPartialStride + 2 + dim] = fmaf(o[i], us, ovrow[r0 + i]);
      }
      tc_fence_before();
      err = named_barrier_or(kGrpBar, kGrp, !ok);
      if (!err && nmore && gt == 0) mbar_arrive(ofree);
    }
    more = (ui.z & 16) == 0;
  }
  if (err && gt == 0) {
    set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
    flags[0] = 1;
  }
  tc_fence_before();
  named_barrier(kFinBar, kFinThreads);
}

// Two forms of the merge of a segment's CTA partials with log-sum-exp weights, then the
// normalisation. Both build the page prefix once per block before waiting (so while the
// attention grid finishes): the previous grid is the same call's attention kernel, which
// triggers this launch only after its own wait, so every grid before it has completed, and it
// writes nothing but the partials and the error word; the context lengths (read at L2, see
// eff_ctx) are taken before waiting.
//
// combine_rows_kernel, for calls with many (segment, query row) items: one warp per item, lane
// l owns output dims 2l, 2l + 1, 64 + 2l and 64 + 2l + 1 (two 8-byte loads of each partial
// row), chunks of kCombChunkWarp partials in flight together, at most 64 registers a thread
// so that one wave holds 4 blocks per SM.
// combine_kernel, for calls with few items (long segments, so many partials each): one block
// of 128 threads per item, thread d owns dim d, chunks of kCombChunkBlock partials.
// Each chunk is merged against its own maximum, then folded into the item's total.
constexpr int kCombWarps = 8;
constexpr int kCombChunkWarp = 4;
constexpr int kCombChunkBlock = 8;

template <int FMT>
__global__ void __launch_bounds__(kCombWarps * 32, 4) combine_rows_kernel(const AttnParams p) {
  extern __shared__ __align__(16) int cpre[];
  volatile int* flags = cpre + p.B + 1;
  build_prefix(p, FMT, cpre, flags);
  griddep_wait();
  griddep_launch_dependents();
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int R = p.R;
  const long long P = (long long)p.Hkv * cpre[p.B];
  const int n_eff = (int)min((long long)p.n_cta, P);
  const int n_items = p.B * p.Hkv * R;
  for (int item = blockIdx.x * kCombWarps + (threadIdx.x >> 5); item < n_items; item += gridDim.x * kCombWarps) {
    const int seg = item / R, row = item - seg * R;
    const int b = seg / p.Hkv, h = seg - (seg / p.Hkv) * p.Hkv;
    const int np = cpre[b + 1] - cpre[b];
    const long long first_pg = (long long)p.Hkv * cpre[b] + (long long)h * np;
    const int c0 = (int)cta_of(first_pg, P, n_eff), c1 = (int)cta_of(first_pg + np - 1, P, n_eff);
    float M = -INFINITY, lsum = 0.0f;
    float2 alo = make_float2(0.0f, 0.0f), ahi = make_float2(0.0f, 0.0f);
    for (int cb = c0; cb <= c1; cb += kCombChunkWarp) {
      float mv[kCombChunkWarp], lv[kCombChunkWarp];
      float2 xl[kCombChunkWarp], xh[kCombChunkWarp];
#pragma unroll
      for (int k = 0; k < kCombChunkWarp; ++k) {
        if (cb + k <= c1) {
          const float* src = p.partials + ((size_t)(cb + k + seg) * R + row) * kPartialStride;
          mv[k] = src[0];
          lv[k] = src[1];
          xl[k] = *reinterpret_cast<const float2*>(src + 2 + 2 * lane);
          xh[k] = *reinterpret_cast<const float2*>(src + 66 + 2 * lane);
        } else {
          mv[k] = -INFINITY;
          lv[k] = 0.0f;
          xl[k] = xh[k] = make_float2(0.0f, 0.0f);
        }
      }
      float Mc = mv[0];
#pragma unroll
      for (int k = 1; k < kCombChunkWarp; ++k) Mc = fmaxf(Mc, mv[k]);
      if (Mc == -INFINITY) continue;  // nothing visible in this chunk
      float lc = 0.0f;
      float2 cl = make_float2(0.0f, 0.0f), ch = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int k = 0; k < kCombChunkWarp; ++k) {
        const float w = fast_exp2(mv[k] - Mc);
        lc += w * lv[k];
        cl.x += w * xl[k].x;
        cl.y += w * xl[k].y;
        ch.x += w * xh[k].x;
        ch.y += w * xh[k].y;
      }
      if (M == -INFINITY) {
        M = Mc;
        lsum = lc;
        alo = cl;
        ahi = ch;
      } else {
        const float Mn = fmaxf(M, Mc);
        const float so = fast_exp2(M - Mn), sc = fast_exp2(Mc - Mn);
        lsum = lsum * so + lc * sc;
        alo.x = alo.x * so + cl.x * sc;
        alo.y = alo.y * so + cl.y * sc;
        ahi.x = ahi.x * so + ch.x * sc;
        ahi.y = ahi.y * so + ch.y * sc;
        M = Mn;
      }
    }
    const int r = row / p.G, gi = row - (row / p.G) * p.G;
    float* dst = p.out + (((size_t)b * p.S + r) * p.Hq + h * p.G + gi) * kD;
    reinterpret_cast<float2*>(dst)[lane] = make_float2(alo.x / lsum, alo.y / lsum);
    reinterpret_cast<float2*>(dst + 64)[lane] = make_float2(ahi.x / lsum, ahi.y / lsum);
  }
}

template <int FMT>
__global__ void __launch_bounds__(128, 4) combine_kernel(const AttnParams p) {
  extern __shared__ __align__(16) int cpre[];
  volatile int* flags = cpre + p.B + 1;
  build_prefix(p, FMT, cpre, flags);
  griddep_wait();
  griddep_launch_dependents();
  __syncthreads();
  const int R = p.R;
  const int n_items = p.B * p.Hkv * R;
  const long long P = (long long)p.Hkv * cpre[p.B];
  const int n_eff = (int)min((long long)p.n_cta, P);
  const int d = threadIdx.x;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int seg = item / R, row = item - seg * R;
    const int b = seg / p.Hkv, h = seg - (seg / p.Hkv) * p.Hkv;
    const int np = cpre[b + 1] - cpre[b];
    const long long first_pg = (long long)p.Hkv * cpre[b] + (long long)h * np;
    const int c0 = (int)cta_of(first_pg, P, n_eff), c1 = (int)cta_of(first_pg + np - 1, P, n_eff);
    float M = -INFINITY, lsum = 0.0f, a = 0.0f;
    for (int cb = c0; cb <= c1; cb += kCombChunkBlock) {
      float mv[kCombChunkBlock], lv[kCombChunkBlock], av[kCombChunkBlock];
#pragma unroll
      for (int k = 0; k < kCombChunkBlock; ++k) {
        if (cb + k <= c1) {
          const float* src = p.partials + ((size_t)(cb + k + seg) * R + row) * kPartialStride;
          mv[k] = src[0];
          lv[k] = src[1];
          av[k] = src[2 + d];
        } else {
          mv[k] = -INFINITY;
          lv[k] = 0.0f;
          av[k] = 0.0f;
        }
      }
      float Mc = mv[0];
#pragma unroll
      for (int k = 1; k < kCombChunkBlock; ++k) Mc = fmaxf(Mc, mv[k]);
      if (Mc == -INFINITY) continue;  // nothing visible in this chunk
      float lc = 0.0f, ac = 0.0f;
#pragma unroll
      for (int k = 0; k < kCombChunkBlock; ++k) {
        const float w = fast_exp2(mv[k] - Mc);
        lc += w * lv[k];
        ac += w * av[k];
      }
      if (M == -INFINITY) {
        M = Mc;
        lsum = lc;
        a = ac;
      } else {
        const float Mn = fmaxf(M, Mc);
        const float so = fast_exp2(M - Mn), sc = fast_exp2(Mc - Mn);
        lsum = lsum * so + lc * sc;
        a = a * so + ac * sc;
        M = Mn;
      }
    }
    const int r = row / p.G, gi = row - (row / p.G) * p.G;
    p.out[(((size_t)b * p.S + r) * p.Hq + h * p.G + gi) * kD + d] = a / lsum;
  }
}

// Combine launch: a block per item while the items fit in one wave of 4 blocks per SM, else a
// warp per item over at most one wave.
template <int FMT>
cudaError_t launch_combine(cudaLaunchConfig_t& cfg, const AttnParams& p, int sm) {
  const long long items = (long long)p.B * p.Hkv * p.R;
  cfg.dynamicSmemBytes = (p.B + 1 + 4) * sizeof(int);
  if (items <= 4LL * sm) {
    cfg.gridDim = dim3((unsigned)std::max<long long>(1, items), 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    return cudaLaunchKernelEx(&cfg, combine_kernel<FMT>, p);
  }
  cfg.gridDim = dim3((unsigned)std::min<long long>((items + kCombWarps - 1) / kCombWarps, 4LL * sm), 1, 1);
  cfg.blockDim = dim3(kCombWarps * 32, 1, 1);
  return cudaLaunchKernelEx(&cfg, combine_rows_kernel<FMT>, p);
}

struct DevCache {
  int sm = 0;
  bool attr[2][4] = {{false}};
  bool tc_attr[4] = {false, false, false, false};  // attn_tc_kernel<24 / 32 / 40 / 48>: shared-memory attribute set
  size_t occ_smem[2][4] = {{0}};  // occupancy cache: last (smem, threads) queried per instantiation
  int occ_threads[2][4] = {{0}};
  int occ[2][4] = {{0}};
};
DevCache g_dev[64];
std::mutex g_dev_mu;  // guards g_dev (launch-configuration caches shared by host threads)

template <int FMT, int NT>
cudaError_t launch_attn_t(AttnParams& p, size_t smem, int threads, long long p_max, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e = cudaSuccess;
  int occ = 1, sm = 1;
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DevCache& dc = g_dev[(dev >= 0 && dev < 64) ? dev : 0];
    if (dc.sm == 0) {
      int n = 0;
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      dc.sm = n > 0 ? n : 1;
    }
    if (!dc.attr[FMT][NT]) {
      e = cudaFuncSetAttribute(attn_kernel<FMT, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
      if (e != cudaSuccess) return e;
      dc.attr[FMT][NT] = true;
    }
    if (dc.occ_smem[FMT][NT] != smem || dc.occ_threads[FMT][NT] != threads) {
      int o = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, attn_kernel<FMT, NT>, threads, smem);
      if (e != cudaSuccess) return e;
      dc.occ[FMT][NT] = std::max(o, 1);
      dc.occ_smem[FMT][NT] = smem;
      dc.occ_threads[FMT][NT] = threads;
    }
    occ = dc.occ[FMT][NT];
    sm = dc.sm;
  }
  long long grid = std::min<long long>((long long)sm * occ, kMaxCtas);
  grid = std::max<long long>(1, std::min(grid, p_max));
  p.n_cta = (int)grid;
  // both grids may start while the previous one on the stream finishes (each waits for it
  // before reading anything)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_kernel<FMT, NT>, p);
  if (e != cudaSuccess) return e;
  return launch_combine<FMT>(cfg, p, sm);
}

// int4 with more than 8 query rows per KV head: the tcgen05 kernel (NR = rows rounded up to 8),
// one CTA per SM (it takes all 512 tensor-memory columns), then the same combine.
template <int NR>
cudaError_t launch_tc_t(AttnParams& p, long long p_max, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = TcLayout(p.B).total + 1024;  // + alignment to 1024 bytes
  cudaError_t e = cudaSuccess;
  int sm = 1;
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DevCache& dc = g_dev[(dev >= 0 && dev < 64) ? dev : 0];
    if (dc.sm == 0) {
      int n = 0;
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      dc.sm = n > 0 ? n : 1;
    }
    static_assert(NR >= 24 && NR <= 48 && NR % 8 == 0, "attn_tc_kernel row counts: 24, 32, 40, 48");
    if (!dc.tc_attr[NR / 8 - 3]) {
      e = cudaFuncSetAttribute(attn_tc_kernel<NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if (e != cudaSuccess) return e;
      dc.tc_attr[NR / 8 - 3] = true;
    }
    sm = dc.sm;
  }
  long long grid = std::min<long long>((long long)sm, kMaxCtas);
  grid = std::max<long long>(1, std::min(grid, p_max));
  p.n_cta = (int)grid;
  p.ntg = 1;
  p.nkg = 1;
  p.nstages = kTcStages;
  p.rows_pad = NR;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<NR>, p);
  if (e != cudaSuccess) return e;
  return launch_combine<0>(cfg, p, sm);
}

}  // namespace

std::atomic<unsigned long long> g_stage_wait_ns{kWaitLimitNs};

void set_stage_wait_limit_ns(unsigned long long ns) { g_stage_wait_ns.store(ns, std::memory_order_relaxed); }

size_t workspace_qrot_bytes(int B, int S, int Hq) { return align_up((size_t)B * S * Hq * kD * 4, 256); }

size_t workspace_partials_bytes(int B, int S, int Hq, int Hkv) {
  const int G = Hq / Hkv;
  return align_up(((size_t)kMaxCtas + (size_t)B * Hkv) * S * G * kPartialStride * 4, 256);
}

cudaError_t launch_attention(const AttnJob& job, cudaStream_t stream) {
  AttnParams p{};
  p.stage_wait_ns = g_stage_wait_ns.load(std::memory_order_relaxed);
  p.B = job.B;
  p.S = job.S;
  p.Hq = job.Hq;
  p.Hkv = job.Hkv;
  p.G = job.Hq / job.Hkv;
  p.R = p.S * p.G;
  p.ctx = job.ctx;
  p.out = job.out;
  p.partials = job.partials;
  p.dev_err = job.dev_err;
  long long p_max;
  if (job.fmt == 0) {
    p.blocks = job.cache.pages;
    p.block_table = job.cache.block_table;
    p.max_pages = job.cache.max_pages_per_seq;
    p.num_pages = job.cache.num_pages;
    p.q_rot = job.q_rot;
    p.score_scale = job.sm_scale * kLog2e;
    p_max = (long long)p.Hkv * p.B * p.max_pages;
  } else {
    p.blocks = job.ring.data;
    p.cap = job.ring.capacity;
    p.window = job.window;
    p.v_scale = job.v_scale;
    p.q = job.q;
    p.q_bf16 = job.q_bf16;
    p.score_scale = job.sm_scale * kLog2e * job.k_scale;
    p_max = (long long)p.Hkv * p.B * (p.cap / kPage);
  }
  const int ntiles = (p.R + 7) / 8;
  if (job.fmt == 0 && p.R > kTcMinRows) {
    switch ((p.R + 7) / 8) {
      case 3: return launch_tc_t<24>(p, p_max, stream);
      case 4: return launch_tc_t<32>(p, p_max, stream);
      case 5: return launch_tc_t<40>(p, p_max, stream);
      default: return launch_tc_t<48>(p, p_max, stream);
    }
  }
  int NT;
  if (ntiles <= 3) {
    NT = ntiles;
    p.ntg = 1;
    p.nkg = NT == 1 ? KVQ_TOKEN_GROUPS : (job.fmt == 0 ? KVQ_TILES3_TOKEN_GROUPS : 4);
    p.nstages = NT == 1 ? KVQ_STAGES_INT4 : (job.fmt == 0 ? KVQ_TILES3_STAGES : 8);
  } else {
    NT = (ntiles + 1) / 2;
    p.ntg = 2;
    p.nkg = job.fmt == 0 ? KVQ_TILES6_TOKEN_GROUPS : 2;
    p.nstages = job.fmt == 0 ? KVQ_TILES6_STAGES : 4;
  }
  if (job.fmt == 1) {  // window rings too large for one cluster per (sequence, KV head)
    p.nkg = NT == 1 ? 4 : 2;
    p.nstages = 4;
  }
  p.rows_pad = p.ntg * NT * 8;
  if (p.nstages % p.nkg != 0) return cudaErrorInvalidConfiguration;  // see the static_assert above
  const int threads = (p.ntg * p.nkg + 1) * 32;
  const SmemLayout L(job.fmt, p.nstages, p.B, p.nkg, p.rows_pad);
  const size_t smem = L.total;
  if (job.fmt == 0) {
    switch (NT) {
      case 1: return launch_attn_t<0, 1>(p, smem, threads, p_max, stream);
      case 2: return launch_attn_t<0, 2>(p, smem, threads, p_max, stream);
      default: return launch_attn_t<0, 3>(p, smem, threads, p_max, stream);
    }
  }
  switch (NT) {
    case 1: return launch_attn_t<1, 1>(p, smem, threads, p_max, stream);
    case 2: return launch_attn_t<1, 2>(p, smem, threads, p_max, stream);
    default: return launch_attn_t<1, 3>(p, smem, threads, p_max, stream);
  }
}

}  // namespace kvq
