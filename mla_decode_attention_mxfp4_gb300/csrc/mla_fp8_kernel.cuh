// Attention kernel for KV stored as fp8 (e4m3) with one per-tensor scale (kernelindex
// "amd-mixed-mla" 676098 "_aiter_mla_decode" and 717900 "_decode": the pages' production path,
// K[t][d] = kv[t][d] * kv_scale, V = K[:, :512]), for sm_103a.
//
// The tensor cores read e4m3 directly, so this kernel has no dequant group: per 96-token tile
// the producer warp brings the 576-byte rows into shared memory with five TMA tensor copies of
// 96 rows x 128 bytes (the 128-byte swizzle; the last copy runs past the row and is zero-filled),
// and the MMA warp runs QK^T with A = that tile (K-major) and P.V with A = the same tile read as
// V^T (MN-major): the operand layouts of the two products coincide for these boxes.  Tiles of
// 96 rows let three stages fit beside the query operands; QK^T keeps M = 128, and its rows
// 96..127 read the next box (finite data, their scores are masked) while P.V sums over the 96
// rows only.  The partition, the query operand (two e4m3 terms per head) and the merge of split sequences are
// those of the MXFP4 path; the softmax is the same online softmax with P' = 2^11 P as two e5m2
// terms, the scores scaled by the per-head factor times kv_scale.  Rows of a tile past its
// sequence get -inf scores by selection, and their V rows are zeroed in shared memory before
// P.V (the rows the copies brought there belong to other sequences and may hold anything).
//
// Warps: 0 MMA issue (and tensor-memory allocation), 1 producer, 2..5 softmax (one per tensor-
// memory lane quarter, 32 tokens each, all 16 heads).
#pragma once
#include <cuda.h>

#include "mla_kernels.cuh"

namespace mla {
namespace fp8 {

constexpr int kTile = 96;    // tokens per tile: three stages fit beside the query operands
constexpr int kMmaM = 128;   // M of the MMAs: QK^T rows 96..127 read the next box and are masked
constexpr int kBoxBytes = 128;                        // inner extent of one copy = the swizzle span
constexpr int kBoxes = (kDqk + kBoxBytes - 1) / kBoxBytes;  // 5: dims 0..639, 576.. zero-filled
constexpr int kVBoxes = kDv / kBoxBytes;              // 4: the V part
constexpr int kBoxTileBytes = kTile * kBoxBytes;      // 12288
constexpr int kStageBytes = kBoxes * kBoxTileBytes;   // 61440
constexpr int kStages = 3;
constexpr int kPrefetch = 2;  // lookahead of the L2 prefetch in tiles (see the producer)
constexpr int kSmWarps = 4;
constexpr int kSmThreads = kSmWarps * 32;
constexpr int kMmaWarp = 0, kProdWarp = 1, kSmWarp0 = 2;
constexpr int kThreads = (2 + kSmWarps) * 32;

// Tensor memory: S^T ring of two (32 columns each: hi query part 0..15, lo part 16..31), two O^T
// accumulators (segment j uses the one at kColO + kColsO (j & 1); each 4 blocks of 128 dims x 32
// columns: P' hi part 0..15, lo part 16..31), so that a segment's output is read while the
// next segment's P.V already accumulates.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 64;
constexpr uint32_t kColsO = 128;

// Shared memory.
constexpr int kOffStages = 0;                                      // boxes 1024-byte aligned
constexpr int kOffQhat = kOffStages + kStages * kStageBytes;       // 184320: [2] query operands
constexpr int kOffPt = kOffQhat + 2 * kQhatBytes;                  // 221184: [2] P^T
constexpr int kOffHmax = kOffPt + 2 * kPtBytes;                    // [2][16 heads][4 quarters]
constexpr int kOffLw = kOffHmax + 2 * 4 * kHeads * 4;              // [16 heads][4 quarters]
constexpr int kOffMlast = kOffLw + 4 * kHeads * 4;                 // [16] output factors
constexpr int kOffMst = kOffMlast + kHeads * 4;                    // [4 warps][16 m, 16 alpha]
constexpr int kOffTmem = kOffMst + 4 * 2 * kHeads * 4;             // tensor-memory address, abort word
constexpr int kOffBar = kOffTmem + 16;
constexpr int kNumBars = 2 * kStages + 6;
constexpr int kSmemBytes = kOffBar + kNumBars * 8;
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kOffQhat % 1024 == 0 && kOffPt % 16 == 0, "operand alignment");

constexpr uint32_t kBarSm = 1;   // softmax group
constexpr uint32_t kBarAll = 2;  // softmax group + MMA warp

struct Fp8Params {
  const float* kv_scale;  // device pointer to the per-tensor scale
  __nv_bfloat16* out;
  Workspace ws;
  int B;
  int rmode;              // kRowModePlain or kRowModeContig
  unsigned long long timeout_ns;
};

__device__ __forceinline__ volatile int* abort_word_fp8() {
  return reinterpret_cast<volatile int*>(dyn_smem + kOffTmem + 4);
}
__device__ __noinline__ void flag_timeout_fp8(int* status) {
  *abort_word_fp8() = 1;
  atomicOr(status, kDeviceTimeout);
}
// Bounded wait (as in the MXFP4 kernel): gives up after timeout_ns, raises MLA_DEVICE_TIMEOUT
// and the abort word; later waits of the thread are single tests.
__device__ __forceinline__ bool wait_fp8(uint64_t* bar, uint32_t parity, const Fp8Params& p, bool& aborted) {
  if (aborted) return mbar_try_wait(bar, parity);
  if (mbar_wait(bar, parity, p.timeout_ns)) return true;
  aborted = true;
  flag_timeout_fp8(&p.ws.meta[kMetaStatus]);
  return false;
}

__global__ void __launch_bounds__(kThreads, 1) mla_split_fp8_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                    const Fp8Params p) {
  uint8_t* smem = dyn_smem;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* bar_full = bars;                     // [kStages] stage landed (producer, tx bytes)
  uint64_t* bar_empty = bars + kStages;          // [kStages] stage read by QK^T and P.V (MMA commit)
  uint64_t* bar_qfree = bars + 2 * kStages;      // [2] query operand buffer read by its segment's last QK^T
  uint64_t* bar_qk = bars + 2 * kStages + 2;     // [2] S^T buffer written (MMA commit)
  uint64_t* bar_pready = bars + 2 * kStages + 4; // P^T written, invalid V rows zeroed, O^T rescaled (softmax)
  uint64_t* bar_pv = bars + 2 * kStages + 5;     // P.V of a tile completed (MMA commit)
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_qfree[0], 1);
    mbar_init(&bar_qfree[1], 1);
    mbar_init(&bar_qk[0], 1);
    mbar_init(&bar_qk[1], 1);
    mbar_init(bar_pready, kSmWarps);
    mbar_init(bar_pv, 1);
    fence_barrier_init();
    *abort_word_fp8() = 0;
  }
  if (warp == kProdWarp && lane == 0) prefetch_tensormap(&tmap);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  grid_dependency_wait();  // the partition kernel's results
  grid_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  TileIterT<kTile> it;
  if (!it.init(p.ws.ipc, p.B, p.ws.cta_desc[2 * g], p.ws.cta_desc[2 * g + 1])) {
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
    return;
  }
  bool aborted = false;

  // =========================== producer warp ===================================
  if (warp == kProdWarp) {
    if (lane != 0) return;
    const uint64_t pol_kv = policy_evict_first();
    const uint64_t pol_q = policy_evict_last();
    // The stages (3 x 60 KB) hold too few bytes in flight to cover the load latency, so when tile
    // k is copied, tile k + kPrefetch (which must wait for a stage) is prefetched into L2: its
    // copy, once a stage is free, then reads L2.
    TileIterT<kTile> pf = it;
    bool pf_ok = true;
    for (int u = 0; u < kPrefetch && pf_ok; ++u) pf_ok = pf.next();
    int k = 0;
    do {
      const int s = k % kStages;
      if (k >= kStages && !wait_fp8(&bar_empty[s], ((k / kStages) - 1) & 1, p, aborted)) break;
      const int j = it.seg;
      if (it.first && j >= 2 && !wait_fp8(&bar_qfree[j & 1], ((j >> 1) - 1) & 1, p, aborted)) break;
      uint8_t* st = smem + kOffStages + s * kStageBytes;
      const int row0 = it.t0 + (p.rmode == kRowModeContig ? p.ws.phys[it.b] - p.ws.ipc[it.b] : 0);
      mbar_arrive_expect_tx(&bar_full[s], (uint32_t)kStageBytes + (it.first ? (uint32_t)kQhatBytes : 0u));
#pragma unroll
      for (int x = 0; x < kBoxes; ++x) tma_load_2d(st + x * kBoxTileBytes, &tmap, x * kBoxBytes, row0, &bar_full[s], pol_kv);
      if (it.first)
        bulk_g2s(smem + kOffQhat + (j & 1) * kQhatBytes, p.ws.qhat + (long long)it.b * kQhatBytes, kQhatBytes,
                 &bar_full[s], pol_q);
      if (pf_ok) {  // pf: tile k + kPrefetch
        const int r = pf.t0 + (p.rmode == kRowModeContig ? p.ws.phys[pf.b] - p.ws.ipc[pf.b] : 0);
#pragma unroll
        for (int x = 0; x < kBoxes; ++x) tma_prefetch_2d(&tmap, x * kBoxBytes, r);
        pf_ok = pf.next();
      }
      ++k;
    } while (!*abort_word_fp8() && it.next());
    for (int s = 0; s < kStages && s < k; ++s) {  // drain: no copy may still be writing at exit
      const int kl = s + ((k - 1 - s) / kStages) * kStages;
      mbar_wait(&bar_full[s], (uint32_t)(kl / kStages) & 1u, p.timeout_ns);
    }
    return;
  }

  // =========================== MMA warp =========================================
  // QK(0); then per tile k: QK(k+1) once its stage landed, P.V(k) once P^T(k) is ready; the
  // stage of tile k is released after P.V(k) (the commit covers QK(k), issued earlier).
  if (warp == kMmaWarp) {
    const uint32_t idesc_qk = idesc_f8(kMmaM, 32, kFmtE4M3, kFmtE4M3, false, false);
    const uint32_t idesc_pv = idesc_f8(kMmaM, 32, kFmtE4M3, kFmtE5M2, true, true);
    const uint64_t dq0 = smem_desc_kmajor(smem_u32(smem + kOffQhat), kQLbo, kQSbo);
    const uint64_t dp0 = smem_desc_mnmajor(smem_u32(smem + kOffPt), kPtLbo, kPtSbo);
    TileIterT<kTile> cur = it, nxt = it;
    bool has_next = nxt.next();
    int k = 0;
    uint64_t* last_bar = nullptr;
    uint32_t last_par = 0;
    for (int kk = 0;; ++kk) {
      if (*abort_word_fp8()) break;
      if (kk == 0 || has_next) {
        const int q = kk;
        const TileIterT<kTile>& qt = kk == 0 ? cur : nxt;
        const int s = q % kStages;
        if (!wait_fp8(&bar_full[s], (q / kStages) & 1, p, aborted)) break;
        tc_fence_after();
        const uint32_t st = smem_u32(smem + kOffStages + s * kStageBytes);
        const uint64_t dq = dq0 + (uint64_t)(((qt.seg & 1) * kQhatBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < kDqk / 32; ++ks) {
          // K-major, 128-byte swizzle: box ks / 4, 32-byte step ks % 4 inside its rows
          const uint64_t da = smem_desc_sw128(st + (ks >> 2) * kBoxTileBytes + (ks & 3) * 32, 16, 1024);
          umma_f8_ss_warp(tmem + kColS + 32 * (q & 1), da, dq + (uint64_t)((ks * 2 * kQLbo) >> 4), idesc_qk,
                          ks > 0 ? 1u : 0u);
        }
        umma_commit_warp(&bar_qk[q & 1]);
        last_bar = &bar_qk[q & 1];
        last_par = (uint32_t)(q >> 1) & 1u;
        if (qt.last) {
          umma_commit_warp(&bar_qfree[qt.seg & 1]);
          last_bar = &bar_qfree[qt.seg & 1];
          last_par = (uint32_t)(qt.seg >> 1) & 1u;
        }
      }
      if (kk == 0) continue;
      if (!wait_fp8(bar_pready, k & 1, p, aborted)) break;
      tc_fence_after();
      const int s = k % kStages;
      const uint32_t st = smem_u32(smem + kOffStages + s * kStageBytes);
      const uint64_t dp = dp0 + (uint64_t)(((k & 1) * kPtBytes) >> 4);
      const bool seg_first = cur.first;
#pragma unroll
      for (int js = 0; js < kTile / 32; ++js)
#pragma unroll
        for (int blk = 0; blk < kVBoxes; ++blk) {
          // V^T, MN-major, 128-byte swizzle: box blk holds dims 128 blk.., 32 tokens = 4 atoms
          const uint64_t da = smem_desc_sw128(st + blk * kBoxTileBytes + js * 32 * kBoxBytes, kBoxTileBytes, 1024);
          umma_f8_ss_warp(tmem + kColO + kColsO * (cur.seg & 1) + 32 * blk, da, dp + (uint64_t)((js * 4 * kPtLbo) >> 4), idesc_pv,
                          (js > 0 || !seg_first) ? 1u : 0u);
        }
      umma_commit_warp(bar_pv);
      umma_commit_warp(&bar_empty[s]);
      last_bar = &bar_empty[s];
      last_par = (uint32_t)(k / kStages) & 1u;
      if (!has_next) break;
      cur = nxt;
      has_next = nxt.next();
      ++k;
    }
    named_sync(kBarAll, kSmThreads + 32);
    if (last_bar) mbar_wait(last_bar, last_par, p.timeout_ns);
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
    return;
  }

  // =========================== softmax group (warps 2..5) =========================
  const int q4 = warp & 3;
  const int t = q4 * 32 + lane;  // token of the tile = tensor-memory lane
  const uint32_t t_lane = tmem + ((uint32_t)(q4 * 32) << 16);
  const int sw = warp - kSmWarp0;
  const int stid = tid - kSmWarp0 * 32;
  float* mstate = reinterpret_cast<float*>(smem + kOffMst) + sw * 2 * kHeads;  // [16] m - kPExp, [16] alpha
  const float kvs = *p.kv_scale;
  float ch[16];  // score factor of each head for the current segment: qch * kv_scale
  float l_part[16];
  // a segment's output waits for the next tile (see the epilogue)
  bool epi = false;
  int epi_b = 0, epi_slot = 0, epi_par = 0;
  bool epi_whole = false;
  auto write_out = [&](int b, int slot, bool whole, int par) {
    const float* ofac = reinterpret_cast<const float*>(smem + kOffMlast);
    float of[16];
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const float4 f4 = *reinterpret_cast<const float4*>(ofac + i);
      of[i] = f4.x; of[i + 1] = f4.y; of[i + 2] = f4.z; of[i + 3] = f4.w;
    }
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      uint32_t a[16], c[16];
      const uint32_t col = t_lane + kColO + kColsO * par + 32 * blk;
      tmem_ld16_nowait(col, a);
      tmem_ld16_nowait(col + 16, c);
      tc_wait_ld();
      const int dim = 128 * blk + t;
      if (whole) {
        __nv_bfloat16* o = p.out + (long long)b * kHeads * kDv + dim;
#pragma unroll
        for (int h = 0; h < kHeads; ++h)
          o[h * kDv] = __float2bfloat16_rn((__uint_as_float(a[h]) + __uint_as_float(c[h])) * of[h]);
      } else {
        float* o = p.ws.part_acc + (long long)slot * kHeads * kDv + dim;
#pragma unroll
        for (int h = 0; h < kHeads; ++h) o[h * kDv] = (__uint_as_float(a[h]) + __uint_as_float(c[h])) * of[h];
      }
    }
    tc_fence_before();
  };
  int k = 0;
  bool has_next;
  do {
    const bool valid = t < it.n;
    const bool seg_first = it.first;
    if (seg_first) {
      const float4* c = reinterpret_cast<const float4*>(p.ws.qch + (long long)it.b * kHeads);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 v = c[i];
        ch[4 * i] = v.x * kvs;
        ch[4 * i + 1] = v.y * kvs;
        ch[4 * i + 2] = v.z * kvs;
        ch[4 * i + 3] = v.w * kvs;
      }
    }
    wait_fp8(&bar_qk[k & 1], (k >> 1) & 1, p, aborted);
    tc_fence_after();
    float s2[16];
    float* hmax = reinterpret_cast<float*>(smem + kOffHmax) + (k & 1) * 4 * kHeads;
    {
      uint32_t rh[16], rl[16];
      const uint32_t scol = t_lane + kColS + 32 * (k & 1);
      tmem_ld16_nowait(scol, rh);
      tmem_ld16_nowait(scol + 16, rl);
      tc_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const float2 sum = f2add(make_float2(__uint_as_float(rh[i]), __uint_as_float(rh[i + 1])),
                                 make_float2(__uint_as_float(rl[i]), __uint_as_float(rl[i + 1])));
        const float2 sv = f2mul(sum, make_float2(ch[i], ch[i + 1]));
        // rows past the tile's tokens hold other data (possibly non-finite): select, not add
        s2[i] = valid ? sv.x : -INFINITY;
        s2[i + 1] = valid ? sv.y : -INFINITY;
      }
    }
    float d[16], alpha_v[16];
    float dmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const float4 a = *reinterpret_cast<const float4*>(mstate + i);
      const float2 d0 = f2sub(make_float2(s2[i], s2[i + 1]), make_float2(a.x, a.y));
      const float2 d1 = f2sub(make_float2(s2[i + 2], s2[i + 3]), make_float2(a.z, a.w));
      d[i] = d0.x; d[i + 1] = d0.y; d[i + 2] = d1.x; d[i + 3] = d1.y;
      dmax = fmaxf(dmax, fmaxf(fmaxf(d0.x, d0.y), fmaxf(d1.x, d1.y)));
      alpha_v[i] = alpha_v[i + 1] = alpha_v[i + 2] = alpha_v[i + 3] = 1.f;
    }
    const bool fits = !seg_first && dmax <= (float)(kMaxThresh + kPExp);
    bool resc = false;
    if (!named_sync_and(kBarSm, kSmThreads, fits)) {
      const float wm = warp_reduce16<true>(s2, lane);
      if ((lane & 1) == 0) hmax[(lane >> 1) * 4 + q4] = wm;
      named_sync(kBarSm, kSmThreads);
      {
        const int h = lane >> 1;
        const float4 hm = *reinterpret_cast<const float4*>(hmax + h * 4);
        const float M = fmaxf(fmaxf(hm.x, hm.y), fmaxf(hm.z, hm.w));
        const float mo = mstate[h];
        float mn = mo, alpha = 1.f;
        bool moved = false;
        if (seg_first) {  // mstate holds m - kPExp, so ex2 gives P' = 2^kPExp P
          mn = M - (float)kPExp;
          alpha = 0.f;
        } else if (M > mo + (float)(kPExp + kMaxThresh)) {
          mn = M - (float)kPExp;
          alpha = ex2(mo - mn);
          moved = true;
        }
        resc = __any_sync(0xffffffffu, moved);  // the same in every warp: all compute every head
        __syncwarp();
        if ((lane & 1) == 0) {
          mstate[h] = mn;
          mstate[kHeads + h] = alpha;
        }
        __syncwarp();
      }
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const float4 a = *reinterpret_cast<const float4*>(mstate + i);
        const float4 b = *reinterpret_cast<const float4*>(mstate + kHeads + i);
        const float2 d0 = f2sub(make_float2(s2[i], s2[i + 1]), make_float2(a.x, a.y));
        const float2 d1 = f2sub(make_float2(s2[i + 2], s2[i + 3]), make_float2(a.z, a.w));
        d[i] = d0.x; d[i + 1] = d0.y; d[i + 2] = d1.x; d[i + 3] = d1.y;
        alpha_v[i] = b.x; alpha_v[i + 1] = b.y; alpha_v[i + 2] = b.z; alpha_v[i + 3] = b.w;
      }
    }
    uint32_t phi[4], plo[4];
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const float2 pv = make_float2(ex2(d[i]), ex2(d[i + 1]));
      const float2 lp = make_float2(l_part[i], l_part[i + 1]);
      const float2 ln = seg_first ? pv : f2fma(lp, make_float2(alpha_v[i], alpha_v[i + 1]), pv);
      l_part[i] = ln.x;
      l_part[i + 1] = ln.y;
      const __half2 p16 = __floats2half2_rn(pv.x, pv.y);
      const __nv_fp8x2_storage_t hi2 =
          __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&p16), __NV_SATFINITE, __NV_E5M2);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(hi2, __NV_E5M2);
      const __half2 rest = __hsub2(p16, *reinterpret_cast<const __half2*>(&hr));
      const __nv_fp8x2_storage_t lo2 =
          __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&rest), __NV_SATFINITE, __NV_E5M2);
      if ((i & 2) == 0) {
        phi[i >> 2] = (uint32_t)hi2;
        plo[i >> 2] = (uint32_t)lo2;
      } else {
        phi[i >> 2] |= (uint32_t)hi2 << 16;
        plo[i >> 2] |= (uint32_t)lo2 << 16;
      }
    }
    {
      uint8_t* prow = smem + kOffPt + (k & 1) * kPtBytes + (t >> 3) * kPtLbo + (t & 7) * 16;
      *reinterpret_cast<uint4*>(prow) = make_uint4(phi[0], phi[1], phi[2], phi[3]);
      *reinterpret_cast<uint4*>(prow + kPtSbo) = make_uint4(plo[0], plo[1], plo[2], plo[3]);
    }
    if (!valid && t < kTile) {  // this row of the stage holds another sequence's data: zero its V part
      uint8_t* vrow = smem + kOffStages + (k % kStages) * kStageBytes + t * kBoxBytes;
#pragma unroll
      for (int x = 0; x < kVBoxes; ++x)
#pragma unroll
        for (int c = 0; c < kBoxBytes / 16; ++c)
          *reinterpret_cast<uint4*>(vrow + x * kBoxTileBytes + 16 * c) = make_uint4(0, 0, 0, 0);
    }
    if (k > 0) wait_fp8(bar_pv, (k - 1) & 1, p, aborted);
    tc_fence_after();
    if (resc) {
#pragma unroll 1
      for (int blk = 0; blk < 4; ++blk) {
        const uint32_t col = t_lane + kColO + kColsO * (it.seg & 1) + 32 * blk;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          uint32_t a[8];
          tmem_ld8_nowait(col + 8 * qq, a);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) a[i] = __float_as_uint(__uint_as_float(a[i]) * alpha_v[(8 * qq + i) & 15]);
          tmem_st8(col + 8 * qq, a);
        }
      }
      tc_wait_st();
    }
    fence_proxy_async_smem();  // P^T and the zeroed rows are read by the tensor cores
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_pready);
    if (epi) {  // the previous segment's output (its last P.V, tile k - 1, was waited for above)
      write_out(epi_b, epi_slot, epi_whole, epi_par);
      epi = false;
    }
    if (it.last) {
      // ---- segment epilogue: O = (hi + lo) * kv_scale / l'; O^T is read at the next tile,
      // after this segment's last P.V, while the next segment accumulates in the other O^T ----
      float* lw = reinterpret_cast<float*>(smem + kOffLw);
      float* ofac = reinterpret_cast<float*>(smem + kOffMlast);
      const float ls = warp_reduce16<false>(l_part, lane);
      if ((lane & 1) == 0) lw[(lane >> 1) * 4 + q4] = ls;
      named_sync(kBarSm, kSmThreads);
      const bool whole = it.whole;
      const int slot = 2 * g + (it.seg > 0 ? 1 : 0);
      if (stid < kHeads) {
        const int h = stid;
        const float4 l4 = *reinterpret_cast<const float4*>(lw + h * 4);
        const float L = (l4.x + l4.y) + (l4.z + l4.w);
        if (!whole) p.ws.part_lse[slot * kHeads + h] = mstate[h] + lg2(L);
        ofac[h] = kvs / L;
      }
      named_sync(kBarSm, kSmThreads);
      epi = true;
      epi_b = it.b;
      epi_slot = slot;
      epi_whole = whole;
      epi_par = it.seg & 1;
    }
    has_next = it.next();
    if (epi && !has_next) {  // the CTA's last segment: its output once its last P.V completed
      wait_fp8(bar_pv, k & 1, p, aborted);
      tc_fence_after();
      write_out(epi_b, epi_slot, epi_whole, epi_par);
      epi = false;
    }
    ++k;
  } while (has_next);
  tc_fence_before();
  named_sync(kBarAll, kSmThreads + 32);
}

}  // namespace fp8
}  // namespace mla
