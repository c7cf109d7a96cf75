// MXFP4 MLA decode attention kernels for sm_103a.
//
// What is computed (kernelindex "amd-mixed-mla" 608791 / 676098 / 717900):
// single-token decode of 16 absorbed-MLA query heads (576 = 512 latent + 64
// RoPE dims) against one shared KV head per token stored as MXFP4 (288 packed
// e2m1 bytes + 18 E8M0 block-32 scales per token); V = first 512 dims; softmax
// scale sm_scale; out bf16 [batch,16,512].  The work is split as in
// "flash-decoding" (split-KV partials + log-sum-exp merge, 608791
// mla_reduce_v1_like_kernel / 676098 _mla_reduce_kernel), but the partition is
// built on the device and the per-split arithmetic is organised for GB300:
//
//  1. mla_partition_kernel (1 CTA): sanitises kv_indptr, cuts the concatenated
//     token stream [indptr[0], indptr[B]) into G equal contiguous ranges (one per
//     resident CTA), and records, per sequence, which ranges it touches and where
//     its partial results go.
//  2. mla_split_kernel (G persistent CTAs, 9 warps): each CTA walks its range in
//     tiles of 128 tokens, one segment per sequence it overlaps.
//       warp 8      producer: bulk async copies (packed rows, scale bytes, and the
//                   query rows at a segment start) into a 3-stage smem ring.
//       warps 0..3  per token: E8M0 exponents -> per-token rebased fp16 factors;
//                   QK^T on tensor cores (mma.sync f16, fp32 accumulate) with the
//                   e2m1 codes converted by cvt.e2m1x2; online softmax; P to smem.
//       warps 4..7  P.V on tensor cores for 128 of the 512 V dims each; the V
//                   fragments are built directly from packed bytes (nibble
//                   interleave of token pairs + cvt.e2m1x2 + factor multiply).
//     A segment that is a whole sequence writes bf16 output directly; otherwise
//     it writes a normalised fp32 partial and its log2-sum-exp.
//  3. mla_merge_kernel (one CTA per sequence): merges the partials of split
//     sequences with weights 2^(lse_s - max lse); empty sequences get zeros.
//
// Numerics: K/V elements are formed exactly in fp16 as e2m1 * 2^(s_tb - S_t),
// S_t the largest scale exponent of token t (exact unless a token's blocks span
// more than 2^23); the token factor 2^(S_t - 127) is applied to the fp32 score
// and, rebased against the running maximum R of S_t, to P before P.V.  Q is
// carried in fp16 with a per-head power-of-two prescale (exact for |q| within
// 2^-28 of the head's largest |q|).  Accumulation, softmax and merge are fp32.
#pragma once
#include <climits>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace mla {

constexpr int kHeads = 16;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kPacked = 288;   // bytes per token
constexpr int kNScale = 18;    // scale bytes per token
constexpr int kTile = 128;     // tokens per tile
constexpr int kStages = 3;
constexpr int kThreads = 288;  // 4 QK warps + 4 PV warps + 1 producer warp
constexpr int kMinPerCta = 64; // smallest token range given to one CTA

constexpr int kDeviceBadIndptr = 1;
constexpr int kDeviceTimeout = 2;

// meta[] fields written by the partition kernel
enum MetaField { kMetaN = 0, kMetaPer = 1, kMetaGeff = 2, kMetaStatus = 3, kMetaSlots = 4 };

struct Workspace {
  int* meta;          // [16]
  int* ipc;           // [B+1] sanitised indptr
  int4* seqinfo;      // [B]: first range, last range, partial slot base, -
  int* cta_first;     // [G]: first sequence overlapping range g
  float* part_lse;    // [2G][16]   log2-sum-exp of each partial
  float* part_acc;    // [2G][16][512] normalised partial output
};

// ---- shared-memory map of mla_split_kernel -----------------------------------
constexpr int kStagePackedBytes = kTile * kPacked;                   // 36864
constexpr int kStageScaleBytes = 2432;                               // >= 128*18 + 32, mult of 16
constexpr int kStageBytes = kStagePackedBytes + kStageScaleBytes;    // 39296
constexpr int kQBytes = kHeads * kDqk * 2;                           // 18432 (bf16 rows)
constexpr int kQhatPitch = 584;                                      // halves per head row (+16 B pad)
constexpr int kFacPitch = 18;                                        // halves per token
constexpr int kSPitch = 20;                                          // floats per token

constexpr int kOffStages = 0;
constexpr int kOffQStage = kOffStages + kStages * kStageBytes;            // 117888
constexpr int kOffQhat = kOffQStage + 2 * kQBytes;                        // 154752
constexpr int kOffFac = kOffQhat + kHeads * kQhatPitch * 2;               // 173440
constexpr int kOffS = kOffFac + 2 * kTile * kFacPitch * 2;                // 182656
constexpr int kOffP = kOffS + kTile * kSPitch * 4;                        // 192896
constexpr int kOffResc = kOffP + 2 * kTile * kHeads * 2;                  // 201088
constexpr int kOffEpi = kOffResc + 2 * kHeads * 4;                        // 201216
constexpr int kOffHmax = kOffEpi + 2 * 48 * 4;                            // 201600
constexpr int kOffRw = kOffHmax + 4 * kHeads * 4;                         // 201856
constexpr int kOffCh = kOffRw + 16;                                       // 201872
constexpr int kOffLw = kOffCh + kHeads * 4;                               // 201936
constexpr int kOffBar = kOffLw + 4 * kHeads * 4;                          // 202192
constexpr int kSmemBytes = kOffBar + 8 * 8;                               // 202256

// named barrier ids (0 is __syncthreads)
constexpr uint32_t kBarPFull = 1;   // +parity
constexpr uint32_t kBarPEmpty = 3;  // +parity
constexpr uint32_t kBarQK = 5;      // QK warps only

struct SplitParams {
  const __nv_bfloat16* q;
  const uint8_t* kv;
  const uint8_t* sc;
  __nv_bfloat16* out;
  Workspace ws;
  int B;
  float sm_scale;
  unsigned long long timeout_ns;
};

// ---- tile iterator: identical walk for every role of a CTA --------------------
struct TileIter {
  const int* ipc;
  int B;
  int b;       // sequence of the current segment
  int s1;      // end row of the current segment
  int t0, n;   // current tile rows [t0, t0+n)
  int r1;      // end of the CTA's range
  int seg;     // segment counter
  bool first, last;

  __device__ bool init(const int* ipc_, int B_, int g, int per, int first_seq) {
    ipc = ipc_;
    B = B_;
    const int rbase = ipc[0];
    const int rend = ipc[B];
    const long long r0ll = (long long)rbase + (long long)g * per;
    if (r0ll >= rend) return false;
    const int r0 = (int)r0ll;
    r1 = (int)min((long long)rend, r0ll + per);
    b = first_seq;
    const int sb = ipc[b];
    t0 = max(r0, sb);
    s1 = min(r1, ipc[b + 1]);
    n = min(kTile, s1 - t0);
    seg = 0;
    first = true;
    last = t0 + n >= s1;
    return n > 0;
  }
  __device__ bool next() {
    if (!last) {
      t0 += n;
      n = min(kTile, s1 - t0);
      first = false;
      last = t0 + n >= s1;
      return true;
    }
    do {
      ++b;
    } while (b < B && ipc[b] == ipc[b + 1]);
    if (b >= B || ipc[b] >= r1) return false;
    t0 = ipc[b];
    s1 = min(r1, ipc[b + 1]);
    n = min(kTile, s1 - t0);
    ++seg;
    first = true;
    last = t0 + n >= s1;
    return true;
  }
};

// ---- block-wide scans for the partition kernel (blockDim = 1024) -------------
template <bool kMax>
__device__ __forceinline__ int block_inclusive_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = kMax ? max(v, u) : v + u;
  }
  if (lane == 31) warp_tot[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w = kMax ? max(w, u) : w + u;
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  if (wid > 0) v = kMax ? max(v, warp_tot[wid - 1]) : v + warp_tot[wid - 1];
  total = warp_tot[31];
  __syncthreads();
  return v;
}

// Sanitise kv_indptr, size the ranges, and describe every sequence's splits.
// kv_null: the KV buffers are absent (NULL), so no row may be read.
__global__ void __launch_bounds__(1024) mla_partition_kernel(const int32_t* __restrict__ indptr, int B,
                                                             int G, int kv_null, Workspace ws) {
  __shared__ int warp_tot[32];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  const int hi = kv_null ? 0 : max(indptr[B], 0);
  // ipc[i] = clamp(max(indptr[0..i]), 0, indptr[B]); every row index stays below indptr[B]
  int carry = INT_MIN;
  for (int base = 0; base <= B; base += 1024) {
    const int i = base + tid;
    int v = (i <= B) ? indptr[i] : INT_MIN;
    if (i <= B && (v < 0 || v > hi || (i > 0 && v < indptr[i - 1]))) s_bad = 1;
    int tot;
    int pm = block_inclusive_scan<true>(v, warp_tot, tot);
    pm = max(pm, carry);
    if (i <= B) ws.ipc[i] = min(max(pm, 0), hi);
    carry = max(carry, tot);
    __syncthreads();
  }
  __threadfence_block();
  __syncthreads();
  const int* ipc = ws.ipc;
  const int rbase = ipc[0];
  const int N = ipc[B] - rbase;
  const long long per_ll = max((long long)kMinPerCta, ((long long)N + G - 1) / G);
  const int per = (int)per_ll;
  const int geff = N > 0 ? (int)(((long long)N + per - 1) / per) : 0;
  // per sequence: ranges [f, l] it overlaps; slot base for split sequences
  int run = 0;
  for (int base = 0; base < B; base += 1024) {
    const int b = base + tid;
    int f = 0, l = -1, nsplit = 0;
    if (b < B) {
      const int a0 = ipc[b], a1 = ipc[b + 1];
      if (a1 > a0) {
        f = (a0 - rbase) / per;
        l = (a1 - 1 - rbase) / per;
        nsplit = l - f + 1;
      }
    }
    const int contrib = nsplit >= 2 ? nsplit : 0;
    int tot;
    const int incl = block_inclusive_scan<false>(contrib, warp_tot, tot);
    if (b < B) ws.seqinfo[b] = make_int4(f, l, run + incl - contrib, 0);
    run += tot;
  }
  // first sequence of each range: largest b with ipc[b] <= r0
  for (int g = tid; g < geff; g += 1024) {
    const int r0 = rbase + g * per;
    int lo = 0, hi2 = B - 1;
    while (lo < hi2) {
      const int mid = (lo + hi2 + 1) >> 1;
      if (ipc[mid] <= r0) lo = mid;
      else hi2 = mid - 1;
    }
    ws.cta_first[g] = lo;
  }
  if (tid == 0) {
    ws.meta[kMetaN] = N;
    ws.meta[kMetaPer] = per;
    ws.meta[kMetaGeff] = geff;
    ws.meta[kMetaStatus] = s_bad ? kDeviceBadIndptr : 0;
    ws.meta[kMetaSlots] = run;
  }
}

// ------------------------------------------------------------------------------
__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, const SplitParams& p,
                                             bool& aborted) {
  if (aborted) return mbar_try_wait(bar, parity);
  if (mbar_wait(bar, parity, p.timeout_ns)) return true;
  aborted = true;
  atomicOr(&p.ws.meta[kMetaStatus], kDeviceTimeout);
  return false;
}

__global__ void __launch_bounds__(kThreads, 1) mla_split_kernel(const SplitParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x;
  const int* meta = p.ws.meta;
  const int geff = meta[kMetaGeff];
  if (g >= geff) return;
  const int per = meta[kMetaPer];

  uint64_t* bar_full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* bar_empty = bar_full + kStages;
  uint64_t* bar_qempty = bar_empty + kStages;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 8);
    }
    mbar_init(&bar_qempty[0], 1);
    mbar_init(&bar_qempty[1], 1);
    fence_barrier_init();
  }
  __syncthreads();

  TileIter it;
  const bool any = it.init(p.ws.ipc, p.B, g, per, p.ws.cta_first[g]);
  if (!any) return;  // cannot happen for g < geff
  bool aborted = false;

  // =========================== producer warp ===================================
  if (warp == 8) {
    if (lane != 0) return;
    const uint64_t pol_kv = policy_evict_first();
    const uint64_t pol_q = policy_evict_last();
    const long long scale_end = (long long)p.ws.ipc[p.B] * kNScale;  // bytes of kv_scale in use
    const long long scale_end16 = scale_end & ~15LL;
    int k = 0;
    do {
      const int s = k % kStages;
      if (k >= kStages) wait_or_flag(&bar_empty[s], ((k / kStages) - 1) & 1, p, aborted);
      const int j = it.seg;
      if (it.first && j >= 2) wait_or_flag(&bar_qempty[j & 1], ((j >> 1) - 1) & 1, p, aborted);
      uint8_t* st = smem + kOffStages + s * kStageBytes;
      // scale bytes [18*t0, 18*(t0+n)): 16-byte aligned superset by bulk copy,
      // anything past the last aligned byte of the buffer by plain loads.
      const long long b0 = (long long)it.t0 * kNScale, b1 = (long long)(it.t0 + it.n) * kNScale;
      const long long a0 = b0 & ~15LL;
      long long a1 = (b1 + 15) & ~15LL;
      if (a1 > scale_end16) a1 = scale_end16;
      uint8_t* sdst = st + kStagePackedBytes;
      for (long long x = (a1 > a0 ? a1 : a0); x < b1; ++x) sdst[x - a0] = p.sc[x];
      uint32_t bytes = (uint32_t)it.n * kPacked + (a1 > a0 ? (uint32_t)(a1 - a0) : 0u);
      if (it.first) bytes += kQBytes;
      mbar_arrive_expect_tx(&bar_full[s], bytes);
      bulk_g2s(st, p.kv + (long long)it.t0 * kPacked, (uint32_t)it.n * kPacked, &bar_full[s], pol_kv);
      if (a1 > a0) bulk_g2s(sdst, p.sc + a0, (uint32_t)(a1 - a0), &bar_full[s], pol_kv);
      if (it.first)
        bulk_g2s(smem + kOffQStage + (j & 1) * kQBytes, p.q + (long long)it.b * kHeads * kDqk, kQBytes,
                 &bar_full[s], pol_q);
      ++k;
    } while (it.next());
    return;
  }

  __half* qhat = reinterpret_cast<__half*>(smem + kOffQhat);
  float* ch = reinterpret_cast<float*>(smem + kOffCh);

  // =========================== QK / softmax warps ===============================
  if (warp < 4) {
    const int t = tid;  // token within the tile for per-token work
    const int r = lane >> 2, c = lane & 3;
    float m_run[kHeads], l_part[kHeads];
    int R = 0;
    int k = 0;
    do {
      const int s = k % kStages, par = k & 1, j = it.seg;
      if (k >= 2) named_sync(kBarPEmpty + par, 256);
      wait_or_flag(&bar_full[s], (k / kStages) & 1, p, aborted);
      const uint8_t* st = smem + kOffStages + s * kStageBytes;
      if (it.first) {
        // ---- segment start: per-head prescale exponent and fp16 Q-hat ----
        const __nv_bfloat16* qs = reinterpret_cast<const __nv_bfloat16*>(smem + kOffQStage + (j & 1) * kQBytes);
        {
          const int h = t >> 3, part = t & 7;
          const uint16_t* qb = reinterpret_cast<const uint16_t*>(qs) + h * kDqk + part * 72;
          uint32_t mx = 0;
          for (int d = 0; d < 72; ++d) mx = max(mx, (uint32_t)(qb[d] & 0x7FFFu));
          mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          if (part == 0) {
            int e = 0;
            if (mx != 0 && mx < 0x7F80u) {
              int ex;
              frexpf(__uint_as_float(mx << 16), &ex);
              e = ex - 1 - 14;
            }
            reinterpret_cast<int*>(smem + kOffLw)[h] = e;
            ch[h] = ldexpf(p.sm_scale * 1.4426950408889634f, e);
          }
        }
        named_sync(kBarQK, 128);
        const int* eh = reinterpret_cast<const int*>(smem + kOffLw);
        for (int e2 = t; e2 < kHeads * kDqk / 2; e2 += 128) {
          const int h = e2 / (kDqk / 2);
          const int rem = (e2 % (kDqk / 2)) * 2;  // even slot index within the head row
          const int ks = rem >> 4, slot = rem & 15;
          const int dim = 32 * (ks >> 1) + 8 * ((slot & 7) >> 1) + 4 * (ks & 1) + 2 * (slot >> 3);
          // q * 2^-e as two exact power-of-two products (e in [-147, 113])
          const int e = eh[h], ea = (-e) / 2, eb = -e - ea;
          const float s1 = exp2i(ea), s2 = exp2i(eb);
          const float q0 = __bfloat162float(qs[h * kDqk + dim]) * s1 * s2;
          const float q1 = __bfloat162float(qs[h * kDqk + dim + 1]) * s1 * s2;
          *reinterpret_cast<__half2*>(qhat + h * kQhatPitch + rem) =
              __halves2half2(__float2half_rn(q0), __float2half_rn(q1));
        }
        named_sync(kBarQK, 128);
        if (t == 0) mbar_arrive(&bar_qempty[j & 1]);
#pragma unroll
        for (int h = 0; h < kHeads; ++h) {
          m_run[h] = -INFINITY;
          l_part[h] = 0.f;
        }
        R = 0;
      }
      // ---- per-token scale exponents -> fp16 factors 2^(s_b - S_t) ----
      const bool valid = t < it.n;
      int St = 0;
      float stok = 0.f;
      {
        uint16_t* fac = reinterpret_cast<uint16_t*>(smem + kOffFac) + par * kTile * kFacPitch + t * kFacPitch;
        const uint8_t* sb = st + kStagePackedBytes + (int)(((long long)it.t0 * kNScale) & 15) + t * kNScale;
        uint32_t sv[kNScale];
        if (valid) {
#pragma unroll
          for (int b = 0; b < kNScale; ++b) {
            sv[b] = sb[b];
            St = max(St, (int)sv[b]);
          }
          stok = (St == 255) ? __int_as_float(0x7FC00000) : exp2i(St - 127);
        }
#pragma unroll
        for (int b = 0; b < kNScale; b += 2) {
          uint32_t lo = 0, hi = 0;
          if (valid) {
            lo = __half_as_ushort(__float2half_rn(exp2i((int)sv[b] - St)));
            hi = __half_as_ushort(__float2half_rn(exp2i((int)sv[b + 1] - St)));
          }
          *reinterpret_cast<uint32_t*>(fac + b) = lo | (hi << 16);
        }
      }
      named_sync(kBarQK, 128);
      // ---- S' = Qhat . (K * 2^(s - S_t)) for this warp's 32 tokens ----
      {
        const uint16_t* fac = reinterpret_cast<const uint16_t*>(smem + kOffFac) + par * kTile * kFacPitch;
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
        const int arow = ((lane >> 3) & 1) * 8 + (lane & 7);
        const __half* qa = qhat + arow * kQhatPitch + (lane >> 4) * 8;
#pragma unroll 2
        for (int b = 0; b < kNScale; ++b) {
          uint32_t aA[4], aB[4];
          ldsm_x4(aA, qa + (2 * b) * 16);
          ldsm_x4(aB, qa + (2 * b + 1) * 16);
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            const int tok = warp * 32 + nt * 8 + r;
            const uint32_t w = *reinterpret_cast<const uint32_t*>(st + tok * kPacked + 16 * b + 4 * c);
            const uint32_t f = fac[tok * kFacPitch + b];
            const uint32_t f2 = f | (f << 16);
            uint32_t kf[4];
            e2m1x8_to_f16x8(w, kf);
#pragma unroll
            for (int i = 0; i < 4; ++i) kf[i] = hmul2_u32(kf[i], f2);
            mma_f16_16816(acc[nt], aA, kf[0], kf[1], acc[nt]);
            mma_f16_16816(acc[nt], aB, kf[2], kf[3], acc[nt]);
          }
        }
        float* S = reinterpret_cast<float*>(smem + kOffS);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int tk = warp * 32 + nt * 8 + 2 * c;
          S[tk * kSPitch + r] = acc[nt][0];
          S[(tk + 1) * kSPitch + r] = acc[nt][1];
          S[tk * kSPitch + r + 8] = acc[nt][2];
          S[(tk + 1) * kSPitch + r + 8] = acc[nt][3];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_empty[s]);
      named_sync(kBarQK, 128);
      // ---- online softmax, one token per thread ----
      {
        const float* S = reinterpret_cast<const float*>(smem + kOffS) + t * kSPitch;
        float s2[kHeads];
#pragma unroll
        for (int h4 = 0; h4 < 4; ++h4) {
          const float4 v = *reinterpret_cast<const float4*>(S + 4 * h4);
          s2[4 * h4 + 0] = v.x;
          s2[4 * h4 + 1] = v.y;
          s2[4 * h4 + 2] = v.z;
          s2[4 * h4 + 3] = v.w;
        }
        float* hmax = reinterpret_cast<float*>(smem + kOffHmax);
#pragma unroll
        for (int h = 0; h < kHeads; ++h) {
          s2[h] = valid ? s2[h] * (ch[h] * stok) : -INFINITY;
          const float wm = warp_max_f32(s2[h]);
          if (lane == 0) hmax[warp * kHeads + h] = wm;
        }
        const int rw = __reduce_max_sync(0xffffffffu, valid ? St : 0);
        if (lane == 0) reinterpret_cast<int*>(smem + kOffRw)[warp] = rw;
        named_sync(kBarQK, 128);
        const int* Rw = reinterpret_cast<const int*>(smem + kOffRw);
        const int Rnew = max(max(R, max(Rw[0], Rw[1])), max(Rw[2], Rw[3]));
        const float rs = exp2i(R - Rnew);
        const float ptok = valid ? exp2i(St - Rnew) : 0.f;
        float* resc = reinterpret_cast<float*>(smem + kOffResc) + par * kHeads;
        uint32_t ph[8];
#pragma unroll
        for (int h = 0; h < kHeads; ++h) {
          const float M = fmaxf(fmaxf(hmax[h], hmax[kHeads + h]), fmaxf(hmax[2 * kHeads + h], hmax[3 * kHeads + h]));
          const float mn = fmaxf(m_run[h], M);
          const float alpha = ex2(m_run[h] - mn);
          if (t == h) resc[h] = alpha * rs;
          const float pv = ex2(s2[h] - mn);
          l_part[h] = l_part[h] * alpha + pv;
          m_run[h] = mn;
          const float pp = pv * ptok;
          if (h & 1) {
            ph[h >> 1] |= (uint32_t)__half_as_ushort(__float2half_rn(pp)) << 16;
          } else {
            ph[h >> 1] = (uint32_t)__half_as_ushort(__float2half_rn(pp));
          }
        }
        R = Rnew;
        uint4* prow = reinterpret_cast<uint4*>(smem + kOffP + par * kTile * kHeads * 2 + t * 32);
        const int sw = (t >> 2) & 1;
        prow[sw] = make_uint4(ph[0], ph[1], ph[2], ph[3]);
        prow[sw ^ 1] = make_uint4(ph[4], ph[5], ph[6], ph[7]);
        if (it.last) {
          float* lw = reinterpret_cast<float*>(smem + kOffLw);
          named_sync(kBarQK, 128);  // everyone is done with eh[] (aliases lw)
#pragma unroll
          for (int h = 0; h < kHeads; ++h) {
            float v = l_part[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) lw[warp * kHeads + h] = v;
          }
          named_sync(kBarQK, 128);
          float* epi = reinterpret_cast<float*>(smem + kOffEpi) + (j & 1) * 48;
          if (t < kHeads) epi[t] = lw[t] + lw[kHeads + t] + lw[2 * kHeads + t] + lw[3 * kHeads + t];
          if (t == 0) {
#pragma unroll
            for (int h = 0; h < kHeads; ++h) epi[kHeads + h] = m_run[h];  // m_run is uniform
          }
          if (t == 0) reinterpret_cast<int*>(epi)[32] = R;
        }
      }
      named_arrive(kBarPFull + par, 256);
      ++k;
    } while (it.next());
    // match the P_EMPTY arrivals of the last two tiles
    for (int kk = max(k - 2, 0); kk < k; ++kk) named_sync(kBarPEmpty + (kk & 1), 256);
    return;
  }

  // =========================== P.V warps =========================================
  {
    const int v = warp - 4;
    const int r = lane >> 2, c = lane & 3, n = lane >> 2;
    float acc[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    int k = 0;
    do {
      const int s = k % kStages, par = k & 1, j = it.seg;
      named_sync(kBarPFull + par, 256);
      wait_or_flag(&bar_full[s], (k / kStages) & 1, p, aborted);
      const uint8_t* st = smem + kOffStages + s * kStageBytes;
      if (it.first) {
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
      } else {
        const float* resc = reinterpret_cast<const float*>(smem + kOffResc) + par * kHeads;
        const float ra = resc[r], rb = resc[r + 8];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          acc[i][0] *= ra;
          acc[i][1] *= ra;
          acc[i][2] *= rb;
          acc[i][3] *= rb;
        }
      }
      const uint8_t* pbase = smem + kOffP + par * kTile * kHeads * 2;
      const uint16_t* fac = reinterpret_cast<const uint16_t*>(smem + kOffFac) + par * kTile * kFacPitch;
      const int blkA = 4 * v + (n >> 2), blkB = blkA + 2;
      // A-fragment row address for ldmatrix.trans: matrix mi = lane/8, row = lane%8
      const int mi = lane >> 3, rowi = lane & 7;
#pragma unroll 1
      for (int ks = 0; ks < kTile / 16; ++ks) {
        uint32_t a[4];
        {
          const int tok = 16 * ks + (mi >> 1) * 8 + rowi;
          const int half = (mi & 1) ^ ((tok >> 2) & 1);
          ldsm_x4_trans(a, pbase + tok * 32 + half * 16);
        }
        const int ta = 16 * ks + 2 * c;
        uint32_t xa[2][2], ya[2][2];  // [token pair 0/1 (+8)][word A/B]
        uint32_t fp[2][2];            // factor pairs [token pair][word A/B]
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const int t0 = ta + 8 * pr;
          const uint8_t* row0 = st + t0 * kPacked + 64 * v + 4 * n;
          const uint8_t* row1 = row0 + kPacked;
          const uint32_t a0 = *reinterpret_cast<const uint32_t*>(row0);
          const uint32_t a1 = *reinterpret_cast<const uint32_t*>(row1);
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(row0 + 32);
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(row1 + 32);
          xa[pr][0] = (a0 & 0x0F0F0F0Fu) | ((a1 << 4) & 0xF0F0F0F0u);
          ya[pr][0] = ((a0 >> 4) & 0x0F0F0F0Fu) | (a1 & 0xF0F0F0F0u);
          xa[pr][1] = (b0 & 0x0F0F0F0Fu) | ((b1 << 4) & 0xF0F0F0F0u);
          ya[pr][1] = ((b0 >> 4) & 0x0F0F0F0Fu) | (b1 & 0xF0F0F0F0u);
          fp[pr][0] = (uint32_t)fac[t0 * kFacPitch + blkA] | ((uint32_t)fac[(t0 + 1) * kFacPitch + blkA] << 16);
          fp[pr][1] = (uint32_t)fac[t0 * kFacPitch + blkB] | ((uint32_t)fac[(t0 + 1) * kFacPitch + blkB] << 16);
        }
#pragma unroll
        for (int wd = 0; wd < 2; ++wd) {
          uint32_t x0[4], y0[4], x1[4], y1[4];
          e2m1x8_to_f16x8(xa[0][wd], x0);
          e2m1x8_to_f16x8(ya[0][wd], y0);
          e2m1x8_to_f16x8(xa[1][wd], x1);
          e2m1x8_to_f16x8(ya[1][wd], y1);
#pragma unroll
          for (int jb = 0; jb < 4; ++jb) {
            const int jx = wd * 8 + 2 * jb, jy = jx + 1;
            mma_f16_16816(acc[jx], a, hmul2_u32(x0[jb], fp[0][wd]), hmul2_u32(x1[jb], fp[1][wd]), acc[jx]);
            mma_f16_16816(acc[jy], a, hmul2_u32(y0[jb], fp[0][wd]), hmul2_u32(y1[jb], fp[1][wd]), acc[jy]);
          }
        }
      }
      if (it.last) {
        // ---- segment epilogue ----
        const float* epi = reinterpret_cast<const float*>(smem + kOffEpi) + (j & 1) * 48;
        const int Rf = reinterpret_cast<const int*>(epi)[32];
        const float os = (Rf == 255) ? __int_as_float(0x7FC00000) : exp2i(Rf - 127);
        const float sa = os / epi[r], sb = os / epi[r + 8];
        const int4 si = p.ws.seqinfo[it.b];
        const bool whole = si.x == si.y;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int d0 = 128 * v + 64 * half + 16 * c;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int head = r + 8 * hh;
            const float sc = hh ? sb : sa;
            float vals[16];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              vals[jj] = acc[half * 8 + jj][2 * hh] * sc;
              vals[8 + jj] = acc[half * 8 + jj][2 * hh + 1] * sc;
            }
            if (whole) {
              uint32_t pk[8];
#pragma unroll
              for (int q2 = 0; q2 < 8; ++q2) {
                __nv_bfloat162 bv = __floats2bfloat162_rn(vals[2 * q2], vals[2 * q2 + 1]);
                pk[q2] = *reinterpret_cast<uint32_t*>(&bv);
              }
              uint4* dst = reinterpret_cast<uint4*>(p.out + ((long long)it.b * kHeads + head) * kDv + d0);
              dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            } else {
              const int slot = si.z + (g - si.x);
              float4* dst = reinterpret_cast<float4*>(p.ws.part_acc + ((long long)slot * kHeads + head) * kDv + d0);
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                dst[q4] = make_float4(vals[4 * q4], vals[4 * q4 + 1], vals[4 * q4 + 2], vals[4 * q4 + 3]);
            }
          }
        }
        if (!whole && v == 0 && lane < kHeads) {
          const int slot = si.z + (g - si.x);
          p.ws.part_lse[slot * kHeads + lane] = epi[kHeads + lane] + lg2(epi[lane]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_empty[s]);
      named_arrive(kBarPEmpty + par, 256);
      ++k;
    } while (it.next());
  }
}

// ---- merge of split sequences -------------------------------------------------------
__global__ void __launch_bounds__(256) mla_merge_kernel(__nv_bfloat16* __restrict__ out, Workspace ws, int B) {
  const int b = blockIdx.x;
  if (b >= B) return;
  const int4 si = ws.seqinfo[b];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int a0 = ws.ipc[b], a1 = ws.ipc[b + 1];
  if (a1 <= a0) {  // empty sequence -> zeros
    uint4* o = reinterpret_cast<uint4*>(out + (long long)b * kHeads * kDv);
    for (int i = tid; i < kHeads * kDv / 8; i += 256) o[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const int ns = si.y - si.x + 1;
  if (ns < 2) return;  // written by the split kernel
  const int base = si.z;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int h = warp * 2 + hh;
    float M = -INFINITY;
    for (int i = lane; i < ns; i += 32) M = fmaxf(M, ws.part_lse[(base + i) * kHeads + h]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int i = lane; i < ns; i += 32) L += ex2(ws.part_lse[(base + i) * kHeads + h] - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    float accv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) accv[i] = 0.f;
    for (int i = 0; i < ns; ++i) {
      const float w = ex2(ws.part_lse[(base + i) * kHeads + h] - M);
      const float4* src = reinterpret_cast<const float4*>(ws.part_acc + ((long long)(base + i) * kHeads + h) * kDv + lane * 16);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 x = src[q4];
        accv[4 * q4] += w * x.x;
        accv[4 * q4 + 1] += w * x.y;
        accv[4 * q4 + 2] += w * x.z;
        accv[4 * q4 + 3] += w * x.w;
      }
    }
    const float inv = 1.f / L;
    uint32_t pk[8];
#pragma unroll
    for (int q2 = 0; q2 < 8; ++q2) {
      __nv_bfloat162 bv = __floats2bfloat162_rn(accv[2 * q2] * inv, accv[2 * q2 + 1] * inv);
      pk[q2] = *reinterpret_cast<uint32_t*>(&bv);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + ((long long)b * kHeads + h) * kDv + lane * 16);
    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  }
}

}  // namespace mla
