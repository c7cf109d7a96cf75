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
//  1. mla_partition_kernel: its first CTA sanitises kv_indptr, counts each sequence's
//     tiles, cuts the concatenated token stream [indptr[0], indptr[B]) into G contiguous
//     ranges of whole tiles (one per resident CTA, at most one tile apart in size), and
//     writes one work descriptor per range (partial slots are fixed by range, so the
//     merge derives them from the tile counts); the other CTAs
//     build each sequence's query operand
//     (e4m3 hi/lo parts of the prescaled query, in its shared-memory image) and
//     the per-head score factors.
//  2. mla_split_kernel (G persistent CTAs, one per SM): each CTA walks its range in
//     tiles of 128 tokens, one segment per sequence it overlaps.  Warp roles:
//       warp 0      MMA issue (one elected lane per tcgen05.mma, whole warp
//                   converged) and the tensor-memory allocation;
//       warp 1      producer: bulk async copies (packed rows and scale bytes into a
//                   3-stage smem ring, the sequence's query operand into one of two
//                   buffers at a segment start);
//       warps 2..5  softmax group, one warp per tensor-memory lane quarter (32
//                   tokens), all 16 heads: online softmax of S^T, P as e5m2 hi + lo
//                   parts, rescaling of the O^T accumulator, V^T of the tile from the
//                   K tile in tensor memory into shared memory, segment epilogue;
//       warps 6..17 dequant group, three warps per lane quarter: the K tile as e5m2
//                   into tensor memory (A operand of QK^T, double-buffered), the
//                   score factors at a segment start;
//       warp 18     reference warp: each landed tile's largest scale byte and its
//                   reference exponent, handed to the dequant group with the stage.
//     QK^T (S^T[128 tokens][32] = K . Qhat^T, hi and lo query parts stacked as N)
//     and P.V (O^T[512][32] += V^T . P^T) run on tcgen05 kind::f8f6f4 with fp32
//     accumulators in tensor memory.  The groups hand tiles to each other through
//     mbarriers only, so tile k+1's dequant overlaps tile k's QK^T, softmax and P.V.
//     A segment that is a whole sequence writes bf16 output directly; otherwise
//     it writes a normalised fp32 partial and its log2-sum-exp.
//  3. mla_merge_kernel (four CTAs per sequence, one warp per head): merges the
//     partials of split sequences with weights 2^(lse_s - max lse); empty
//     sequences get zeros.
//
// Numerics: the K/V operand of tile k is e2m1 * 2^(s_tb - R_k + kHead) in e5m2, with R_k the
// tile's reference exponent (its largest scale byte, or a little above it, see
// next_reference) and kHead = 13 the headroom that puts the largest possible element
// (6 * 2^13 = 49152) just under the e5m2 maximum.  Such a value has at most two
// significant bits, so it is exact in e5m2 (the high byte of its fp16 form) for
// s_tb >= R_k - 27; blocks further below are zero.  The tile factor 2^(R_k - 127 - kHead)
// multiplies the fp32 scores, and the O^T accumulator, which holds P.V against the
// reference of the latest tile, is rescaled by 2^(R_old - R_new) when the reference changes.
// The query is q * 2^-E_h (E_h per head) as two e4m3 terms, which hold a bf16 value
// exactly unless it lies more than 2^11 below its head's maximum.  P = 2^(s - m) uses a
// running maximum m that is only raised when a tile's maximum exceeds it by more than
// 2^4, so P <= 16; it enters P.V as two e5m2 terms of 2^11 P (about 6 significant bits for
// every weight down to ~2^-20 of the largest, so long flat tails of small weights are kept).
// Scores, softmax statistics, accumulation and the merge are fp32.
#pragma once
#include <climits>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "ptx.cuh"

namespace mla {

constexpr int kHeads = 16;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kPacked = 288;   // bytes per token
constexpr int kNScale = 18;    // scale bytes per token
constexpr int kTile = 128;     // tokens per tile
constexpr int kStages = 3;
constexpr int kDqWarps = 12;                 // dequant group: 3 warps per tensor-memory lane quarter
constexpr int kDqThreads = kDqWarps * 32;
constexpr int kDqParts = kDqWarps / 4;      // dequant warps per lane quarter
constexpr int kSmWarps = 4;                  // softmax group: 1 warp per lane quarter
constexpr int kSmThreads = kSmWarps * 32;
constexpr int kTokWarps = kDqWarps + kSmWarps;
constexpr int kTokThreads = kTokWarps * 32;
// Warp roles, in warp-index order (lower indices are favoured by the issue
// schedulers, so the latency-critical roles come first): MMA issue, producer,
// softmax group, dequant group, tile references.  A warp reaches tensor-memory lanes
// 32*(warp % 4)..+31; both groups cover every quarter.
constexpr int kMmaWarp = 0;                  // tcgen05.mma issue (also allocates tensor memory)
constexpr int kProdWarp = 1;                 // bulk async copies
constexpr int kSmWarp0 = 2;                  // softmax group: warps 2..5
constexpr int kDqWarp0 = kSmWarp0 + kSmWarps;  // dequant group: warps 6..17
constexpr int kRefWarp = kDqWarp0 + kDqWarps;   // tile reference exponents: warp 18
constexpr int kThreads = (kTokWarps + 3) * 32;
constexpr int kPartSmemSeqs = 8192;  // the partition kernel keeps ipc in shared memory up to this batch
constexpr int kPartMaxGrid = 1024;   // most split CTAs the partition kernel cuts ranges for

constexpr int kDeviceBadIndptr = 1;
constexpr int kDeviceTimeout = 2;

// meta[] fields written by the partition kernel
enum MetaField { kMetaN = 0, kMetaTiles = 1, kMetaGeff = 2, kMetaStatus = 3, kMetaRows = 4 };

// Partial slots: range g's first segment writes slot 2g and its last segment slot 2g + 1
// when they are parts of split sequences (any other segment of a range is a whole
// sequence).  A sequence b split over ranges f..l therefore has its partials in slots
// 2f + (b starts after range f's first row), 2(f+1), ..., 2l.

// "Sequences" below are query rows: with one query row per sequence they are the sequences
// themselves; with several (qo_indptr) each query row is its own problem over its
// sequence's KV rows.  ipc is the prefix of their KV lengths in the logical token stream the
// CTAs split; phys maps a query row's logical rows to physical KV rows.
struct Workspace {
  int* meta;          // [16]
  int* ipc;           // [S+1] logical token offsets (the sanitised kv_indptr in the plain layout)
  int4* cta_desc;     // [G][2]: range g = {r0, r1, first sequence b, ipc[b]}, {ipc[b+1], -, -, -}
  float* part_lse;    // [2G][16]   log2-sum-exp of each partial
  float* part_acc;    // [2G][16][512] normalised partial output
  uint8_t* qhat;      // [S][kQhatBytes] query operand of each sequence, in its shared-memory image
  float* qch;         // [S][16] score factor of each head: sm_scale * log2(e) * 2^E_h
  int* kvc;           // [Bkv+1] sanitised kv_indptr (general layout only)
  int* qoc;           // [Bkv+1] sanitised qo_indptr for more than kPartSmemSeqs sequences (general layout)
  int* phys;          // [S] first physical row, or first entry of kv_indices (general layout only)
  int* tp;            // [S+1] tiles of the split kernel in the sequences before each one
};

// Layout of the KV rows beyond the plain one (kv_indptr rows, one query row per sequence).
struct RowMap {
  const int32_t* qo_indptr;   // [Bkv+1] query rows of each sequence, or null (row b = sequence b)
  const int32_t* kv_indices;  // paged: page ids, kv_indptr counting entries of it; null: kv_indptr counts rows
  const int32_t* last_len;    // paged: rows used in each sequence's last page, [Bkv]
  int Bkv;                    // sequences (kv_indptr holds Bkv + 1 entries)
  int page_size;              // paged: rows per page
  int num_pages;              // paged: pages the KV buffers hold
  int kv_rows;                // > 0: rows the KV buffer holds (kv_indptr is clamped to it, and flagged)
};
constexpr int kRowModePlain = 0, kRowModeContig = 1, kRowModePaged = 2;
// Longer sequences are clamped (and flagged); 1024 of them still sum within int32 in the
// partition kernel's block scan.
constexpr int kMaxRowsPerQuery = 1 << 20;

// ---- shared-memory and tensor-memory map of mla_split_kernel ---------------
constexpr int kStagePackedBytes = kTile * kPacked;                   // 36864
constexpr int kStageScaleBytes = 2432;                               // >= 128*18 + 32, mult of 16
constexpr int kStageBytes = kStagePackedBytes + kStageScaleBytes;    // 39296
// The scale bytes of a tile land in the first 16 + 128*18 bytes of the scale area.  The last
// word holds the offset (0..15) at which the tile's first scale byte landed (written by the
// producer before the stage's copies are announced); the word before it the tile's reference
// exponent R (written by the reference warp once the stage has landed).
constexpr int kStageMisOff = kStagePackedBytes + kStageScaleBytes - 4;
constexpr int kStageRefOff = kStageMisOff - 4;
static_assert(kStageRefOff >= kStagePackedBytes + 16 + ((kTile * kNScale + 15) / 16) * 16, "stage spare words");
constexpr int kQhatBytes = 32 * kDqk;                                // 18432: e4m3 hi + lo query parts

// Tensor memory (32-bit columns, lane = token of the tile / row of M):
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 0;      // 2 x 144 columns: e5m2 K tile, column c = dims 4c..4c+3
constexpr uint32_t kColsA = 144;
constexpr uint32_t kColS = 288;    // 2 x 32 columns: S^T from the hi (0..15) and lo (16..31) query parts
constexpr uint32_t kColSt = 352;   // 4 columns: reference exponent R of the tile (tile k in column k % 4, every lane)
constexpr uint32_t kColO = 384;    // 128 columns: O^T, 4 blocks of 128 dims x (16 hi + 16 lo P parts)

// Qhat, e4m3 hi (n = head) and lo (n = 16 + head) parts, K-major without swizzle:
// offset(n, d) = (d/16)*kQLbo + (n/8)*kQSbo + (n%8)*16 + d%16.
constexpr uint32_t kQLbo = 512, kQSbo = 128;
// V^T, e5m2, MN-major without swizzle, 4 blocks of 128 dims:
// offset(d, t) = (d/128)*kVtBlock + (t/8)*kVtLbo + ((d%128)/16)*kVtSbo + (t%8)*16 + d%16.
constexpr uint32_t kVtBlock = 16384, kVtLbo = 1024, kVtSbo = 128;
// P^T, e5m2, MN-major, two buffers, n = head (hi part) or 16 + head (lo part):
// offset(n, t) = (t/8)*kPtLbo + (n/16)*kPtSbo + (t%8)*16 + n%16.
constexpr uint32_t kPtLbo = 256, kPtSbo = 128, kPtBytes = kTile * 32;
constexpr int kMaxThresh = 4;  // raise the running maxima only by more than this (log2 units)
// Headroom of the K/V operand: a block at the tile's reference exponent is stored as
// e2m1 * 2^kHead, so its largest possible element 6 * 2^13 = 49152 stays below the e5m2
// maximum 57344 and blocks down to 27 binades below the reference stay exact (smallest e5m2
// subnormal: 2^-16).
constexpr int kHead = 13;
constexpr float kHeadInv = 1.f / 8192.f;  // 2^-kHead
static_assert(kHeadInv * (1 << kHead) == 1.f, "headroom factor");
// P enters P.V as two e5m2 terms of P' = 2^kPExp P (hi = e5m2(P') in O^T columns 0..15 of a
// block, lo = e5m2(P' - hi) in columns 16..31): about 6 significant bits for every weight from
// the largest down to ~2^-20 of it (e5m2's exponent range keeps long flat tails of small
// weights).  The softmax keeps its running maxima as m - kPExp, so P' comes out of ex2 directly;
// the row sums then hold 2^kPExp l, and the factor cancels in O / l and in m + log2 l.
constexpr int kPExp = 11;      // P' <= 2^(kPExp + kMaxThresh) = 2^15 < the e5m2 maximum
constexpr float kOutInv = kHeadInv;

constexpr int kOffStages = 0;
constexpr int kOffQhat = kOffStages + kStages * kStageBytes;              // 117888: [2] (segment parity)
constexpr int kOffVt = kOffQhat + 2 * kQhatBytes;                         // 154752
constexpr int kOffPt = kOffVt + 4 * kVtBlock;                             // 220288
constexpr int kOffHmax = kOffPt + 2 * kPtBytes;                           // 228480: [2][16 heads][4 quarters]
constexpr int kOffCh = kOffHmax + 2 * 4 * kHeads * 4;                     // 228992: [4][16] score factors
constexpr int kOffLw = kOffCh + 4 * kHeads * 4;                           // 229248: [16 heads][4 quarters]
constexpr int kOffMlast = kOffLw + 4 * kHeads * 4;                        // 229504: [16] output factors
constexpr int kOffMst = kOffMlast + kHeads * 4;                           // 229568: [4 warps][16 m, 16 alpha]
constexpr int kOffTmem = kOffMst + 4 * 2 * kHeads * 4;                    // 230080: tensor-memory address
constexpr int kOffAbort = kOffTmem + 4;                                   // abort word (bounded waits)
constexpr int kOffBar = kOffTmem + 16;                                    // 230096
constexpr int kNumBars = 20;
constexpr int kOffPid = kOffBar + kNumBars * 8;                           // 230256: [16] page ids of a tile (producer)
constexpr int kTilePidSlots = 16;
constexpr int kSmemBytes = kOffPid + kTilePidSlots * 4;                   // 230320
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kOffVt % 16 == 0 && kOffPt % 16 == 0 && kOffQhat % 16 == 0, "operand alignment");

constexpr uint32_t kBarSm = 1;     // named barrier of the softmax group
constexpr uint32_t kBarAll = 2;    // dequant + softmax groups + MMA warp

struct SplitParams {
  const uint8_t* kv;
  const uint8_t* sc;  // the 16-byte boundary at or below kv_scale (kv_scale = sc + sc_mis)
  int sc_mis;         // kv_scale's offset from that boundary (0..15)
  int rmode;          // kRowMode*: how logical token rows map to physical KV rows
  const int32_t* kv_indices;  // paged: page ids
  int page_size, num_pages;   // paged
  __nv_bfloat16* out;
  Workspace ws;
  int B;
  unsigned long long timeout_ns;
  int stall_producer;  // test hook: the producer issues no copy, so the first wait on a stage gives up
};

// ---- tile iterator: identical walk for every role of a CTA --------------------
template <int kT>
struct TileIterT {
  const int* ipc;
  int B;
  int b;       // sequence of the current segment
  int s1;      // end row of the current segment
  int t0, n;   // current tile rows [t0, t0+n)
  int r1;      // end of the CTA's range
  int seg;     // segment counter
  bool first, last;
  bool whole;  // the current segment is its whole sequence

  // d0 = {r0, r1, first sequence b, ipc[b]}, d1.x = ipc[b+1] (written by the partition kernel)
  __device__ bool init(const int* ipc_, int B_, int4 d0, int4 d1) {
    ipc = ipc_;
    B = B_;
    const int r0 = d0.x;
    r1 = d0.y;
    if (r0 >= r1) return false;
    b = d0.z;
    t0 = max(r0, d0.w);
    s1 = min(r1, d1.x);
    n = min(kT, s1 - t0);
    seg = 0;
    first = true;
    last = t0 + n >= s1;
    whole = d0.w >= r0 && d1.x <= r1;
    return n > 0;
  }
  __device__ bool next() {
    if (!last) {
      t0 += n;
      n = min(kT, s1 - t0);
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
    whole = ipc[b + 1] <= r1;
    n = min(kT, s1 - t0);
    ++seg;
    first = true;
    last = t0 + n >= s1;
    return true;
  }
};
using TileIter = TileIterT<kTile>;

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

// Query operand of one head of one sequence (one warp): per-head prescale exponent E_h,
// score factor sm_scale * log2(e) * 2^E_h, and the e4m3 hi/lo parts of
// Qhat = q * 2^-E_h (two e4m3 terms hold a bf16 value exactly unless it lies more than
// 2^11 below its head's maximum), written as the split kernel's shared-memory image of
// the operand (offset(n, d) of the Qhat layout; n = h for the hi part, 16 + h for the
// lo part) so that one bulk copy lands it.  Lane l converts the 16-dim chunks l and
// l + 32.
__device__ __forceinline__ void build_qhat_head(const __nv_bfloat16* __restrict__ q, float sm_scale, int b, int h,
                                                int lane, const Workspace& ws) {
  const uint4* qr = reinterpret_cast<const uint4*>(q + ((long long)b * kHeads + h) * kDqk);
  constexpr int kChunks = kDqk / 16;  // 36
  uint4 x[2][2];
  uint32_t mx = 0;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int ch = lane + 32 * c;
    if (ch < kChunks) {
      x[c][0] = qr[2 * ch];
      x[c][1] = qr[2 * ch + 1];
      const uint32_t w[8] = {x[c][0].x, x[c][0].y, x[c][0].z, x[c][0].w, x[c][1].x, x[c][1].y, x[c][1].z, x[c][1].w};
#pragma unroll
      for (int i = 0; i < 8; ++i) mx = max(mx, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
    }
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  int e = 0;
  float f = 1.f;
  if (mx >= 0x7F80u) {
    f = __int_as_float(0x7FC00000);  // a non-finite query makes the head's scores NaN
  } else if (mx != 0) {
    int ex;
    frexpf(__uint_as_float(mx << 16), &ex);
    e = ex - 8;  // max |q| * 2^-e in [128, 256): below the e4m3 maximum 448
  }
  if (lane == 0) {
    const int ea = e / 2, eb = e - ea;  // exact 2^e as two factors (e in [-141, 120])
    ws.qch[b * kHeads + h] = sm_scale * 1.4426950408889634f * exp2i(ea) * exp2i(eb) * f;
  }
  const int na = (-e) / 2, nb = -e - na;
  const float s1 = exp2i(na), s2 = exp2i(nb);
  uint8_t* img = ws.qhat + (long long)b * kQhatBytes + (h >> 3) * kQSbo + (h & 7) * 16;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int ch = lane + 32 * c;
    if (ch >= kChunks) continue;
    const uint32_t w[8] = {x[c][0].x, x[c][0].y, x[c][0].z, x[c][0].w, x[c][1].x, x[c][1].y, x[c][1].z, x[c][1].w};
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      uint32_t hw[2], lw[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float q0 = __uint_as_float(w[i + j] << 16) * s1 * s2;
        const float q1 = __uint_as_float(w[i + j] & 0xFFFF0000u) * s1 * s2;
        const __nv_fp8x2_storage_t hi2 = __nv_cvt_float2_to_fp8x2(make_float2(q0, q1), __NV_SATFINITE, __NV_E4M3);
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(hi2, __NV_E4M3);
        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        const __nv_fp8x2_storage_t lo2 =
            __nv_cvt_float2_to_fp8x2(make_float2(q0 - hf.x, q1 - hf.y), __NV_SATFINITE, __NV_E4M3);
        hw[j] = hi2;
        lw[j] = lo2;
      }
      hi[i >> 1] = hw[0] | (hw[1] << 16);
      lo[i >> 1] = lw[0] | (lw[1] << 16);
    }
    *reinterpret_cast<uint4*>(img + ch * kQLbo) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(img + ch * kQLbo + 2 * kQSbo) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// Block 0: sanitise kv_indptr, size the ranges, and describe every sequence's splits.
// kv_null: the KV buffers are absent (NULL), so no row may be read.
// Blocks 1..: the query operand of sequences 2(x-1) and 2(x-1)+1 (warp w: head w % 16),
// so the split kernel copies it instead of building it at every segment start.
// B is the number of query rows (sequences of the logical stream).  With rm.qo_indptr or
// rm.kv_indices set (the general layout), block 0 first derives every query row's KV length
// and physical start from the sequence it belongs to.
constexpr int kPartThreads = 1024;
constexpr int kQhatSeqsPerBlock = kPartThreads / 32 / kHeads;  // 2
__global__ void __launch_bounds__(kPartThreads, 1) mla_partition_kernel(const int32_t* __restrict__ indptr, int B,
                                                                     int G, int kv_null, Workspace ws,
                                                                     const __nv_bfloat16* __restrict__ q,
                                                                     float sm_scale, RowMap rm, int tile) {
  grid_launch_dependents();  // the split kernel's prologue may run alongside
  // Launched with programmatic serialization, this grid may be resident before the
  // preceding kernel in the stream (the previous call's merge kernel, or whatever wrote
  // kv_indptr or q) has finished: wait for it before the first load.
  grid_dependency_wait();
  const int tid = threadIdx.x;
  if (blockIdx.x > 0) {
    const int b = (blockIdx.x - 1) * kQhatSeqsPerBlock + (tid >> 5) / kHeads;
    if (b < B) build_qhat_head(q, sm_scale, b, (tid >> 5) % kHeads, tid & 31, ws);
    return;
  }
  __shared__ int warp_tot[32];
  __shared__ int s_bad;
  __shared__ int s_ipc[kPartSmemSeqs + 1];  // copy of ipc for batch <= kPartSmemSeqs
  __shared__ int s_cut[kPartMaxGrid + 1];   // first row of each range, and the end
  __shared__ int s_first[kPartMaxGrid];     // first sequence of each range
  const bool in_smem = B <= kPartSmemSeqs;
  const bool general = rm.qo_indptr != nullptr || rm.kv_indices != nullptr;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  if (!general) {
    int hi = kv_null ? 0 : max(indptr[B], 0);
    if (rm.kv_rows > 0 && hi > rm.kv_rows) {
      hi = rm.kv_rows;
      if (tid == 0) s_bad = 1;
    }
    // ipc[i] = clamp(max(indptr[0..i]), 0, indptr[B]); every row index stays below indptr[B]
    int carry = INT_MIN;
    for (int base = 0; base <= B; base += 1024) {
      const int i = base + tid;
      int v = (i <= B) ? indptr[i] : INT_MIN;
      if (i <= B && (v < 0 || v > hi || (i > 0 && v < indptr[i - 1]))) s_bad = 1;
      int tot;
      int pm = block_inclusive_scan<true>(v, warp_tot, tot);
      pm = max(pm, carry);
      if (i <= B) {
        const int c = min(max(pm, 0), hi);
        ws.ipc[i] = c;
        if (in_smem) s_ipc[i] = c;
      }
      carry = max(carry, tot);
      __syncthreads();
    }
    if (tid == 0) ws.meta[kMetaRows] = hi;
  } else {
    // 1. kv_indptr over the Bkv sequences -> kvc, sanitised as above (counting rows, or
    //    entries of kv_indices when paged)
    const int Bkv = rm.Bkv;
    const bool paged = rm.kv_indices != nullptr;
    int hi = kv_null ? 0 : max(indptr[Bkv], 0);
    if (!paged && rm.kv_rows > 0 && hi > rm.kv_rows) {
      hi = rm.kv_rows;
      if (tid == 0) s_bad = 1;
    }
    int carry = INT_MIN;
    for (int base = 0; base <= Bkv; base += 1024) {
      const int i = base + tid;
      int v = (i <= Bkv) ? indptr[i] : INT_MIN;
      if (i <= Bkv && (v < 0 || v > hi || (i > 0 && v < indptr[i - 1]))) s_bad = 1;
      int tot;
      int pm = block_inclusive_scan<true>(v, warp_tot, tot);
      pm = max(pm, carry);
      if (i <= Bkv) ws.kvc[i] = min(max(pm, 0), hi);
      carry = max(carry, tot);
      __syncthreads();
    }
    // 2. qo_indptr -> its sanitised copy (shared memory for up to kPartSmemSeqs sequences;
    //    s_ipc is free until step 3 has read it), clamped to [0, B]
    int* qoc = nullptr;
    if (rm.qo_indptr) {
      qoc = Bkv <= kPartSmemSeqs && !in_smem ? s_ipc : ws.qoc;
      carry = INT_MIN;
      for (int base = 0; base <= Bkv; base += 1024) {
        const int i = base + tid;
        int v = (i <= Bkv) ? rm.qo_indptr[i] : INT_MIN;
        if (i <= Bkv && (v < 0 || v > B || (i > 0 && v < rm.qo_indptr[i - 1]))) s_bad = 1;
        int tot;
        int pm = block_inclusive_scan<true>(v, warp_tot, tot);
        pm = max(pm, carry);
        if (i <= Bkv) qoc[i] = min(max(pm, 0), B);
        carry = max(carry, tot);
        __syncthreads();
      }
      if (tid == 0 && (rm.qo_indptr[0] != 0 || rm.qo_indptr[Bkv] != B)) s_bad = 1;
    }
    __threadfence_block();
    __syncthreads();
    // 3. every query row j: its sequence, KV length and physical start; ipc = exclusive prefix
    //    of the lengths (rows past the total that int32 offsets can hold get length 0)
    long long lcarry = 0;
    for (int base = 0; base < B + 1024; base += 1024) {
      if (base > B) break;
      const int j = base + tid;
      int len = 0, ph = 0, b = -1;
      if (j < B) {
        if (qoc) {  // the last sequence whose first query row is <= j, if j lies inside it
          int lo = 0, hi2 = Bkv - 1;
          while (lo < hi2) {
            const int mid = (lo + hi2 + 1) >> 1;
            if (qoc[mid] <= j) lo = mid;
            else hi2 = mid - 1;
          }
          b = (Bkv > 0 && qoc[lo] <= j && j < qoc[lo + 1]) ? lo : -1;
        } else {
          b = j < Bkv ? j : -1;
        }
        if (b >= 0) {
          const int k0 = ws.kvc[b], k1 = ws.kvc[b + 1];
          if (paged) {
            const int np = k1 - k0;
            int last = 0;
            if (np > 0) {
              last = rm.last_len[b];
              if (last < 1 || last > rm.page_size) {
                s_bad = 1;
                last = min(max(last, 1), rm.page_size);
              }
            }
            const long long L = np > 0 ? (long long)(np - 1) * rm.page_size + last : 0;
            len = (int)min(L, (long long)kMaxRowsPerQuery);
            if (L > kMaxRowsPerQuery) s_bad = 1;
          } else {
            len = min(k1 - k0, kMaxRowsPerQuery);
            if (k1 - k0 > kMaxRowsPerQuery) s_bad = 1;
          }
          ph = k0;
        }
      }
      __syncthreads();  // every row's qoc lookups are done before s_ipc (possibly holding qoc) is rewritten
      int tot;
      const int incl = block_inclusive_scan<false>(len, warp_tot, tot);
      const long long start = lcarry + incl - len;
      if (j <= B) {
        const int c = (int)min(start, (long long)INT_MAX);
        ws.ipc[j] = c;
        if (in_smem) s_ipc[j] = c;
        if (start > INT_MAX) s_bad = 1;
      }
      if (j < B) ws.phys[j] = ph;
      lcarry += tot;
      __syncthreads();
    }
    if (tid == 0) ws.meta[kMetaRows] = paged ? (int)min((long long)rm.num_pages * rm.page_size, (long long)INT_MAX) : hi;
  }
  __threadfence_block();
  __syncthreads();
  const int* ipc = in_smem ? s_ipc : ws.ipc;
  const int rbase = ipc[0];
  const int N = ipc[B] - rbase;
  // Tiles: each sequence is walked in tiles of `tile` rows from its first row, the last one
  // possibly short; tp[b] counts the tiles of the sequences before b.  A tile costs the split
  // kernel the same time however many of its rows are used, so the ranges are cut in whole
  // tiles: range g gets tiles [x_g, x_{g+1}), x_g = floor(g T / geff), geff = min(G, T).
  int T = 0;
  for (int base = 0; base <= B; base += 1024) {
    const int i = base + tid;
    const int nt = i < B ? (ipc[i + 1] - ipc[i] + tile - 1) / tile : 0;
    int tot;
    const int incl = block_inclusive_scan<false>(nt, warp_tot, tot);
    if (i <= B) ws.tp[i] = T + incl - nt;
    T += tot;
  }
  const int geff = min(G, T);
  __threadfence_block();
  __syncthreads();
  // the first row of each range and its first sequence: range g starts in the sequence whose
  // tiles hold x_g, at row ipc[b] + (x_g - tp[b]) tile
  for (int b = tid; b < B; b += 1024) {
    const int t0 = ws.tp[b], t1 = ws.tp[b + 1];
    if (t1 <= t0) continue;
    const int g0 = (int)(((long long)t0 * geff + T - 1) / T), g1 = (int)(((long long)t1 * geff + T - 1) / T);
    for (int g = g0; g < g1; ++g) {
      const int x = (int)((long long)g * T / geff);
      s_cut[g] = ipc[b] + (x - t0) * tile;
      s_first[g] = b;
    }
  }
  if (tid == 0) s_cut[geff] = rbase + N;
  __syncthreads();
  // per range: its rows, its first sequence and that sequence's rows, so a CTA starts from
  // one 32-byte load; empty ranges have r0 == r1
  for (int g = tid; g < G; g += 1024) {
    int4 d0 = make_int4(0, 0, 0, 0), d1 = make_int4(0, 0, 0, 0);
    if (g < geff) {
      const int lo = s_first[g];
      d0 = make_int4(s_cut[g], s_cut[g + 1], lo, ipc[lo]);
      d1.x = ipc[lo + 1];
    }
    ws.cta_desc[2 * g] = d0;
    ws.cta_desc[2 * g + 1] = d1;
  }
  if (tid == 0) {
    ws.meta[kMetaN] = N;
    ws.meta[kMetaTiles] = T;
    ws.meta[kMetaGeff] = geff;
    ws.meta[kMetaStatus] = s_bad ? kDeviceBadIndptr : 0;
  }
}

// ------------------------------------------------------------------------------
// Bounded wait of the split kernel: gives up after p.timeout_ns of global time, raises
// MLA_DEVICE_TIMEOUT in the status word and sets the CTA's abort word.  After that every
// wait of the thread is a single test, so the CTA runs to its end without blocking: the
// roles keep their control flow (every named barrier is still reached by all its warps),
// and the producer and the MMA warp, which read the abort word once per tile, issue no
// further asynchronous work and drain what they issued.
// The abort word lives at a fixed offset of the dynamic shared memory; addressed through the
// symbol, its address is a constant (no pointer kept live across the kernel).
extern __shared__ __align__(1024) uint8_t dyn_smem[];
__device__ __forceinline__ volatile int* abort_word() {
  return reinterpret_cast<volatile int*>(dyn_smem + kOffAbort);
}
// The failure path, out of line (it runs at most once per thread).
__device__ __noinline__ void flag_timeout(int* status) {
  *abort_word() = 1;
  atomicOr(status, kDeviceTimeout);
}
__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, const SplitParams& p,
                                             bool& aborted) {
  if (aborted) return mbar_try_wait(bar, parity);
  if (mbar_wait(bar, parity, p.timeout_ns)) return true;
  aborted = true;
  flag_timeout(&p.ws.meta[kMetaStatus]);
  return false;
}

// f16 2^r as the bit pattern of an f16x2 pair: exponent field r + 15 when normal, a
// subnormal bit down to 2^-24, else 0 (r <= 0).
__device__ __forceinline__ uint32_t f16x2_pow2(int r) {
  const uint32_t hb = r >= -14 ? (uint32_t)(r + 15) << 10 : (r >= -24 ? 1u << (r + 24) : 0u);
  return hb * 0x10001u;
}
// 32 e2m1 codes (one 16-byte chunk) times an f16x2 factor -> 32 e5m2 bytes.
__device__ __forceinline__ void chunk_to_e5m2(const uint4 w, uint32_t f2, uint32_t (&e)[8]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v[4];
    e2m1x8_to_f16x8(ws[i], v);
    e[2 * i] = f16x4_hi_bytes(hmul2_u32(v[0], f2), hmul2_u32(v[1], f2));
    e[2 * i + 1] = f16x4_hi_bytes(hmul2_u32(v[2], f2), hmul2_u32(v[3], f2));
  }
}

// Reference exponent of tile k: R_k = T_k, the largest scale byte of the tile, at a segment
// start or when T_k exceeds the previous reference; the previous reference while T_k stays
// within kRefSlack below it (no accumulator rescale for small steps down); never more than
// kRefDrop below the largest reference of the segment so far, so that accumulated values
// stay within fp32 range when they are expressed against a much lower reference.
constexpr int kRefSlack = 4;
constexpr int kRefDrop = 64;
__device__ __forceinline__ int next_reference(int T, int r_prev, int r_max, bool seg_first) {
  if (seg_first || T > r_prev) return T;
  if (T < r_prev - kRefSlack) return max(T, r_max - kRefDrop);
  return r_prev;
}

// K tile -> tensor memory as e5m2 against the tile reference R (one exponent for every token
// of the tile): K[t][d] = e2m1 * 2^(s_tb - R + kHead).  R >= every scale byte of the tile, so
// the largest possible element is 6 * 2^13, below the e5m2 maximum; a block is exact for
// s_tb >= R - 27 (its fp16 factor 2^(s_tb - R + 13) is a normal number down to 2^-14, and every
// product is then a normal or subnormal e5m2 value with a zero low byte in fp16); blocks
// further below are zero.  Tokens past the tile are zero.  Token t = this thread's lane of
// the quarter; part p converts the consecutive blocks 6p .. 6p+5, two per step (the next
// pair's bytes are loaded while this pair is converted; one 16-column store per pair).
// Part 0 stores R in tensor-memory column r_col for the softmax group.
__device__ __forceinline__ void k_tile_to_tmem(const uint8_t* st, int n, int t, int part, uint32_t a_lane,
                                               uint32_t r_col, int R) {
  const bool valid = t < n;
  // where the tile's first scale byte landed (0..15): the producer's note in the stage, masked
  // so that a stage that never landed (a wait that gave up) is still read in bounds
  const int mis = *reinterpret_cast<const int*>(st + kStageMisOff) & 15;
  const uint8_t* sb = st + kStagePackedBytes + mis + t * kNScale;
  constexpr int kNb = kNScale / kDqParts;  // consecutive blocks b0 .. b0 + kNb - 1 of this part
  static_assert(kNScale % kDqParts == 0 && kNb % 2 == 0, "pairs of blocks per part");
  const int b0 = part * kNb;
  const uint8_t* sp = sb + b0;
  if (part == 0) {
    const uint32_t rv[1] = {(uint32_t)R};
    tmem_st1(r_col, rv);
  }
  // f16 exponent field of 2^(s - R + kHead) is s + sbias when positive
  const int sbias = valid ? 15 + kHead - R : -1024;
  const uint8_t* row = st + t * kPacked + 16 * b0;
  uint4 wa = *reinterpret_cast<const uint4*>(row), wb = *reinterpret_cast<const uint4*>(row + 16);
  // not unrolled: the warp roles of a CTA share the instruction caches
#pragma unroll 1
  for (int j = 0; j < kNb; j += 2) {
    const uint4 xa = wa, xb = wb;
    if (j + 2 < kNb) {
      wa = *reinterpret_cast<const uint4*>(row + 16 * j + 32);
      wb = *reinterpret_cast<const uint4*>(row + 16 * j + 48);
    }
    const int ta = sp[j], tb = sp[j + 1];
    uint32_t e[16];
    chunk_to_e5m2(xa, (uint32_t)max(ta + sbias, 0) * 0x04000400u, *reinterpret_cast<uint32_t(*)[8]>(&e[0]));
    chunk_to_e5m2(xb, (uint32_t)max(tb + sbias, 0) * 0x04000400u, *reinterpret_cast<uint32_t(*)[8]>(&e[8]));
    tmem_st16(a_lane + 8 * (b0 + j), e);
  }
}

// Maximum (kMax) or sum over the 32 lanes of sixteen per-lane values; lane L ends
// with the result for value index L >> 1.
template <bool kMax>
__device__ __forceinline__ float warp_reduce16(const float (&v)[16], int lane) {
  float a[8], c[4], d[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // lanes with bit 4 keep values 8..15
    const float send = b4 ? v[i] : v[i + 8], keep = b4 ? v[i + 8] : v[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 16);
    a[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b3 ? a[i] : a[i + 4], keep = b3 ? a[i + 4] : a[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 8);
    c[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b2 ? c[i] : c[i + 2], keep = b2 ? c[i + 2] : c[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 4);
    d[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
  float x;
  {
    const float send = b1 ? d[0] : d[1], keep = b1 ? d[1] : d[0];
    const float r = __shfl_xor_sync(0xffffffffu, send, 2);
    x = kMax ? fmaxf(keep, r) : keep + r;
  }
  const float r1 = __shfl_xor_sync(0xffffffffu, x, 1);
  return kMax ? fmaxf(x, r1) : x + r1;
}

// Reference warp of mla_split_kernel (out of line: its registers stay apart from the other
// roles').  It walks the tiles in the producer's order: once a stage has landed, the warp
// takes the tile's largest scale byte T over its tokens and the tile's reference exponent R
// (next_reference), leaves R in the stage and signals the dequant group.
__device__ __noinline__ void reference_warp(uint8_t* smem, uint64_t* bar_full, uint64_t* bar_tready, TileIter it,
                                            uint64_t timeout_ns, int* status, int lane) {
  int r_prev = 0, r_max = 0;  // reference of the last tile, largest of its segment so far
  for (int k = 0;; ++k) {
    const int s = k % kStages;
    if (*abort_word()) break;
    if (!__all_sync(0xffffffffu, mbar_wait(&bar_full[s], (uint32_t)(k / kStages) & 1u, timeout_ns))) {
      if (lane == 0) flag_timeout(status);
      break;
    }
    uint8_t* st = smem + kOffStages + s * kStageBytes;
    const int lo = *reinterpret_cast<const int*>(st + kStageMisOff) & 15;
    const int hi = lo + it.n * kNScale;  // the tile's scale bytes are [lo, hi) of the scale area
    uint32_t acc = 0;                    // maxima of the even and the odd bytes, as 16-bit lanes
    for (int c = lane; 16 * c < hi; c += 32) {
      const uint4 w4 = *reinterpret_cast<const uint4*>(st + kStagePackedBytes + 16 * c);
      const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int o = 16 * c + 4 * i;
        uint32_t m = 0xFFFFFFFFu;
        if (o < lo || o + 4 > hi) {  // a word at either end: only bytes in [lo, hi) count
          m = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            if (o + b >= lo && o + b < hi) m |= 0xFFu << (8 * b);
        }
        const uint32_t v = ws[i] & m;
        acc = vmax_u16x2(acc, prmt(v, 0u, 0x4240u));
        acc = vmax_u16x2(acc, prmt(v, 0u, 0x4341u));
      }
    }
    const int T = (int)__reduce_max_sync(0xffffffffu, max(acc & 0xFFFFu, acc >> 16));
    const int R = next_reference(T, r_prev, r_max, it.first);
    r_max = it.first ? R : max(r_max, R);
    r_prev = R;
    __syncwarp();
    if (lane == 0) {
      *reinterpret_cast<int*>(st + kStageRefOff) = R;
      mbar_arrive(&bar_tready[s]);
    }
    if (!it.next()) break;
  }
}

// O^T rescale (out of line: it runs only when a running maximum or the tile reference
// moves): column 8q + i of each block holds head (8q + i) % 16, scaled by alpha[head] * rs.
__device__ __noinline__ void rescale_o(uint32_t t_lane, const float* alpha, float rs) {
  float f[16];
#pragma unroll
  for (int i = 0; i < 16; i += 4) {
    const float4 a4 = *reinterpret_cast<const float4*>(alpha + i);
    f[i] = a4.x * rs; f[i + 1] = a4.y * rs; f[i + 2] = a4.z * rs; f[i + 3] = a4.w * rs;
  }
#pragma unroll 1
  for (int blk = 0; blk < 4; ++blk) {
    const uint32_t col = t_lane + kColO + 32 * blk;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t a[8];
      tmem_ld8_nowait(col + 8 * q, a);
      tc_wait_ld();
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = __float_as_uint(__uint_as_float(a[i]) * f[(8 * q + i) & 15]);
      tmem_st8(col + 8 * q, a);
    }
  }
  tc_wait_st();
}

// Segment output (out of line: it runs once per segment, apart from the per-tile code):
// O^T of the thread's dims (t + 128 blk), times each head's factor, as bf16 output rows
// (whole sequences) or fp32 partial rows.
__device__ __noinline__ void segment_out(void* dst, bool whole, const float* ofac, uint32_t t_lane, int t) {
  float of[16];
#pragma unroll
  for (int i = 0; i < 16; i += 4) {
    const float4 f4 = *reinterpret_cast<const float4*>(ofac + i);
    of[i] = f4.x; of[i + 1] = f4.y; of[i + 2] = f4.z; of[i + 3] = f4.w;
  }
#pragma unroll 1
  for (int blk = 0; blk < 4; ++blk) {
    uint32_t a[16], c[16];
    const uint32_t col = t_lane + kColO + 32 * blk;
    tmem_ld16_nowait(col, a);
    tmem_ld16_nowait(col + 16, c);
    tc_wait_ld();
    const int dim = 128 * blk + t;
    if (whole) {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(dst) + dim;
#pragma unroll
      for (int h = 0; h < kHeads; ++h)
        o[h * kDv] = __float2bfloat16_rn(((__uint_as_float(a[h]) + __uint_as_float(c[h])) * kOutInv) * of[h]);
    } else {
      float* o = static_cast<float*>(dst) + dim;
#pragma unroll
      for (int h = 0; h < kHeads; ++h) o[h * kDv] = ((__uint_as_float(a[h]) + __uint_as_float(c[h])) * kOutInv) * of[h];
    }
  }
}

// Producer warp of mla_split_kernel, one thread (out of line, like the reference warp: its
// code lies apart from the other roles').  It walks the tiles in the CTA's order and fills
// stage k % kStages once the dequant group released it: packed rows and scale bytes by bulk
// copies, and the sequence's query operand into buffer (segment & 1) at a segment start.
__device__ __noinline__ void producer_warp(uint8_t* smem, const SplitParams& pp, TileIter it, uint64_t* bar_full,
                                           uint64_t* bar_empty, uint64_t* bar_qfree) {
  const SplitParams p = pp;  // the fields in registers
  bool aborted = false;
  const uint64_t pol_kv = policy_evict_first();
  const uint64_t pol_q = policy_evict_last();
  // scale byte x of physical row r is at sc[sc_mis + 18r]; the bytes in use end at scale_end, and
  // the buffer's first 16-byte boundary is head16
  const long long scale_end = p.sc_mis + (long long)p.ws.meta[kMetaRows] * kNScale;
  const long long scale_end16 = scale_end & ~15LL;
  const long long head16 = (p.sc_mis + 15) & ~15LL;
  // Paged layout: the run of the tile's tokens that starts at tile row i lies in one page:
  // `cnt` rows from physical row `row`.
  // Paged layout: the sequence's logical start and its first kv_indices entry are loaded
  // once per segment; a tile's page ids (at most kTilePidSlots of them when page_size >= 9)
  // are loaded together and kept in shared memory while one pass walks the runs.
  int* pid_s = reinterpret_cast<int*>(smem + kOffPid);
  int seg_b = -1, seg_pos0 = 0, seg_ix0 = 0;
  int k = 0;
  if (!p.stall_producer) do {
    const int s = k % kStages;
    if (k >= kStages && !wait_or_flag(&bar_empty[s], ((k / kStages) - 1) & 1, p, aborted)) break;
    const int j = it.seg;
    // segment j's Qhat goes to buffer j & 1 once the last QK^T of segment j - 2 read it
    if (it.first && j >= 2 && !wait_or_flag(&bar_qfree[j & 1], ((j >> 1) - 1) & 1, p, aborted))
      break;
    uint8_t* st = smem + kOffStages + s * kStageBytes;
    uint8_t* sdst = st + kStagePackedBytes;
    if (p.rmode != kRowModePaged) {
      // one run of rows from physical row row0 (row0 = t0 in the plain layout)
      const long long row0 =
          it.t0 + (p.rmode == kRowModeContig ? (long long)p.ws.phys[it.b] - p.ws.ipc[it.b] : 0LL);
      // the tile's scale bytes [b0, b1) land at stage offset x - a0 (a0 = b0 rounded down to 16):
      // the 16-byte chunks inside the buffer [c0, a1) by bulk copy, the bytes before the
      // buffer's first boundary and past its last one by plain loads
      const long long b0 = p.sc_mis + row0 * kNScale, b1 = b0 + (long long)it.n * kNScale;
      const long long a0 = b0 & ~15LL;
      const long long c0 = a0 > head16 ? a0 : head16;
      long long a1 = (b1 + 15) & ~15LL;
      if (a1 > scale_end16) a1 = scale_end16;
      for (long long x = b0; x < b1 && x < c0; ++x) sdst[x - a0] = p.sc[x];
      for (long long x = (a1 > c0 ? a1 : c0); x < b1; ++x) sdst[x - a0] = p.sc[x];
      *reinterpret_cast<int*>(st + kStageMisOff) = (int)(b0 & 15);
      uint32_t bytes = (uint32_t)it.n * kPacked + (a1 > c0 ? (uint32_t)(a1 - c0) : 0u);
      if (it.first) bytes += kQhatBytes;
      mbar_arrive_expect_tx(&bar_full[s], bytes);
      bulk_g2s(st, p.kv + row0 * kPacked, (uint32_t)it.n * kPacked, &bar_full[s], pol_kv);
      if (a1 > c0) bulk_g2s(sdst + (c0 - a0), p.sc + c0, (uint32_t)(a1 - c0), &bar_full[s], pol_kv);
    } else {
      // Paged: one run per page the tile touches.  A run's scale bytes [g0, g1) land at stage
      // offset dst0 + (x - g0), dst0 = M + 18 i: the 16-byte chunks [c0, a1) by bulk copy when
      // source and destination agree modulo 16, the other bytes by plain loads.  At the tile's
      // own ends the bulk range may round outwards (the extra bytes land outside the tile's
      // part of the area); between runs it rounds inwards.  One pass over the runs issues the
      // plain loads and the bulk copies and counts the bulk bytes; the stage is announced with
      // that count afterwards (the barrier's transaction count may run below zero until then,
      // and the phase cannot complete before this thread's arrival).
      if (it.b != seg_b) {
        seg_b = it.b;
        seg_pos0 = p.ws.ipc[seg_b];
        seg_ix0 = p.ws.phys[seg_b];
      }
      const int ps = p.page_size;
      const int pos0 = it.t0 - seg_pos0;
      const int pg0 = pos0 / ps, off0 = pos0 - pg0 * ps;
      const int npg = (off0 + it.n + ps - 1) / ps;  // pages the tile touches
      const bool in_smem = npg <= kTilePidSlots;
      auto clamp_page = [&](int page) {  // an id outside the buffers is clamped into them, and flagged
        if (page < 0 || page >= p.num_pages) {
          atomicOr(&p.ws.meta[kMetaStatus], kDeviceBadIndptr);
          page = min(max(page, 0), max(p.num_pages - 1, 0));
        }
        return page;
      };
      if (in_smem) {
        const int* src = p.kv_indices + seg_ix0 + pg0;
        int u = 0;
        for (; u + 4 <= npg; u += 4) {  // four loads in flight, then their stores
          const int a0 = src[u], a1v = src[u + 1], a2 = src[u + 2], a3 = src[u + 3];
          pid_s[u] = clamp_page(a0);
          pid_s[u + 1] = clamp_page(a1v);
          pid_s[u + 2] = clamp_page(a2);
          pid_s[u + 3] = clamp_page(a3);
        }
        for (; u < npg; ++u) pid_s[u] = clamp_page(src[u]);
      }
      int M = 0;
      uint32_t bytes = it.first ? (uint32_t)kQhatBytes : 0u;
      for (int u = 0; u < npg; ++u) {
        // run u: tile rows [i, i + cnt) from physical row `row`
        const int page = in_smem ? pid_s[u] : clamp_page(p.kv_indices[seg_ix0 + pg0 + u]);
        const int off = u == 0 ? off0 : 0;
        const int i = u == 0 ? 0 : ps * u - off0;
        const int cnt = min(ps - off, it.n - i);
        const long long row = (long long)page * ps + off;
        const long long g0 = p.sc_mis + row * kNScale, g1 = g0 + (long long)cnt * kNScale;
        if (u == 0) M = (int)(g0 & 15);
        const long long dst0 = M + (long long)i * kNScale;
        long long c0 = g1, a1 = g1;  // no bulk range
        if (((g0 - dst0) & 15) == 0) {
          c0 = i == 0 ? (g0 & ~15LL) : ((g0 + 15) & ~15LL);
          a1 = i + cnt == it.n ? ((g1 + 15) & ~15LL) : (g1 & ~15LL);
          if (c0 < head16) c0 = head16;
          if (a1 > scale_end16) a1 = scale_end16;
          if (a1 < c0) a1 = c0;
        }
        for (long long x = g0; x < g1 && x < c0; ++x) sdst[dst0 + (x - g0)] = p.sc[x];
        for (long long x = (a1 > g0 ? a1 : g0); x < g1; ++x) sdst[dst0 + (x - g0)] = p.sc[x];
        bytes += (uint32_t)cnt * kPacked + (uint32_t)(a1 - c0);
        bulk_g2s(st + i * kPacked, p.kv + row * kPacked, (uint32_t)cnt * kPacked, &bar_full[s], pol_kv);
        if (a1 > c0) bulk_g2s(sdst + dst0 + (c0 - g0), p.sc + c0, (uint32_t)(a1 - c0), &bar_full[s], pol_kv);
      }
      *reinterpret_cast<int*>(st + kStageMisOff) = M;
      mbar_arrive_expect_tx(&bar_full[s], bytes);
    }
    if (it.first)
      bulk_g2s(smem + kOffQhat + (j & 1) * kQhatBytes, p.ws.qhat + (long long)it.b * kQhatBytes, kQhatBytes,
               &bar_full[s], pol_q);
    ++k;
  } while (!*abort_word() && it.next());
  // Drain before this warp leaves: the last phase issued on each stage completes once its
  // copies have landed (in a normal run the dequant group has waited for all of them; after
  // an abort it may not have, and no copy may still be writing when the CTA exits).
  for (int s = 0; s < kStages && s < k; ++s) {
    const int kl = s + ((k - 1 - s) / kStages) * kStages;  // last tile issued on stage s
    mbar_wait(&bar_full[s], (uint32_t)(kl / kStages) & 1u, p.timeout_ns);
  }
}

__global__ void __launch_bounds__(kThreads, 1) mla_split_kernel(const __grid_constant__ SplitParams p) {
  uint8_t* smem = dyn_smem;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* bar_full = bars;          // [3] stage landed (producer, tx bytes)
  uint64_t* bar_empty = bars + 3;     // [3] stage consumed (dequant group)
  uint64_t* bar_qfree = bars + 6;     // [2] Qhat buffer b read by the last QK^T of its segment (MMA commit)
  uint64_t* bar_kready = bars + 8;    // [2] K tile in tensor-memory buffer b ready, its Qhat landed (dequant group)
  // (slot 10 unused)
  uint64_t* bar_pready = bars + 11;   // [2] P^T and V^T of tile k and any O^T rescale done (softmax group)
  uint64_t* bar_qk = bars + 13;       // [2] S^T buffer b written (MMA commit); its tile's R_k is in tensor memory
  uint64_t* bar_pv = bars + 15;       // [2] P.V of tile k completed (barrier k & 1; MMA commit)
  uint64_t* bar_tready = bars + 17;   // [3] stage landed and its tile's reference exponent written (reference warp)
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], kDqWarps);
    }
    mbar_init(&bar_qfree[0], 1);
    mbar_init(&bar_qfree[1], 1);
    mbar_init(&bar_kready[0], kDqWarps);
    mbar_init(&bar_kready[1], kDqWarps);
    mbar_init(&bar_pready[0], kSmWarps);
    mbar_init(&bar_pready[1], kSmWarps);
    mbar_init(&bar_qk[0], 1);
    mbar_init(&bar_qk[1], 1);
    mbar_init(&bar_pv[0], 1);
    mbar_init(&bar_pv[1], 1);
    for (int s = 0; s < kStages; ++s) mbar_init(&bar_tready[s], 1);
    fence_barrier_init();
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  if (tid == 0) *abort_word() = 0;
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
  // Everything above overlaps the partition kernel (programmatic dependent launch); its
  // results are read from here on.  The merge kernel may be scheduled from now on: it waits
  // for this grid's completion itself.
  grid_dependency_wait();
  grid_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  TileIter it;
  if (!it.init(p.ws.ipc, p.B, p.ws.cta_desc[2 * g], p.ws.cta_desc[2 * g + 1])) {  // a range beyond the tokens
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
    return;
  }
  bool aborted = false;

  // =========================== producer warp ===================================
  if (warp == kProdWarp) {
    if (lane != 0) return;
    producer_warp(smem, p, it, bar_full, bar_empty, bar_qfree);
    return;
  }

  // =========================== reference warp ===================================
  if (warp == kRefWarp) {
    reference_warp(smem, bar_full, bar_tready, it, p.timeout_ns, &p.ws.meta[kMetaStatus], lane);
    return;
  }

  // =========================== MMA warp =========================================
  // Order of issue: QK(0), then per tile k: QK(k+1) once its K tile is ready, P.V(k) once the
  // softmax group has written its P^T and V^T.  QK(k+1) follows P.V(k-1), which follows the
  // softmax of tile k-1 (the last reader of the S^T buffer that QK(k+1) writes).
  if (warp == kMmaWarp) {
    const uint32_t idesc_qk = idesc_f8(kTile, 32, kFmtE5M2, kFmtE4M3, false, false);
    const uint32_t idesc_pv = idesc_f8(kTile, 32, kFmtE5M2, kFmtE5M2, true, true);
    const uint64_t dq0 = smem_desc_kmajor(smem_u32(smem + kOffQhat), kQLbo, kQSbo);
    const uint64_t dv0 = smem_desc_mnmajor(smem_u32(smem + kOffVt), kVtLbo, kVtSbo);
    const uint64_t dp0 = smem_desc_mnmajor(smem_u32(smem + kOffPt), kPtLbo, kPtSbo);
    // the last commit issued: it arrives once every MMA issued before it has completed
    uint64_t* last_bar = nullptr;
    uint32_t last_par = 0;
    auto issue_qk = [&](int q, const TileIter& qt) {
      tc_fence_after();
      const uint32_t bq = q & 1;
      const uint64_t dq = dq0 + (uint64_t)(((qt.seg & 1) * kQhatBytes) >> 4);
#pragma unroll
      for (int ks = 0; ks < kDqk / 32; ++ks)
        umma_f8_ts_warp(tmem + kColS + 32 * bq, tmem + kColA + kColsA * bq + 8 * ks,
                        dq + (uint64_t)((ks * 2 * kQLbo) >> 4), idesc_qk, ks > 0 ? 1u : 0u);
      umma_commit_warp(&bar_qk[bq]);
      last_bar = &bar_qk[bq];
      last_par = (uint32_t)(q >> 1) & 1u;
      if (qt.last) {  // the segment's Qhat buffer may be refilled
        umma_commit_warp(&bar_qfree[qt.seg & 1]);
        last_bar = &bar_qfree[qt.seg & 1];
        last_par = (uint32_t)(qt.seg >> 1) & 1u;
      }
    };
    auto issue_pv = [&](int k, bool seg_first) {
      tc_fence_after();
      const uint64_t dp = dp0 + (uint64_t)(((k & 1) * kPtBytes) >> 4);
#pragma unroll
      for (int js = 0; js < kTile / 32; ++js)
#pragma unroll
        for (int blk = 0; blk < 4; ++blk)
          umma_f8_ss_warp(tmem + kColO + 32 * blk, dv0 + (uint64_t)((blk * kVtBlock + js * 4 * kVtLbo) >> 4),
                          dp + (uint64_t)((js * 4 * kPtLbo) >> 4), idesc_pv, (js > 0 || !seg_first) ? 1u : 0u);
      umma_commit_warp(&bar_pv[k & 1]);
      last_bar = &bar_pv[k & 1];
      last_par = (uint32_t)(k >> 1) & 1u;
    };
    TileIter cur = it, nxt = it;  // tiles k and k+1
    bool has_next = nxt.next();
    if (!*abort_word() && wait_or_flag(&bar_kready[0], 0, p, aborted)) {
      issue_qk(0, cur);
      for (int k = 0;; ++k) {
        bool qk_todo = has_next, pv_todo = true;
        if (*abort_word()) break;
        if (has_next) {
          if (!wait_or_flag(&bar_kready[(k + 1) & 1], ((k + 1) >> 1) & 1, p, aborted)) break;
          issue_qk(k + 1, nxt);
          qk_todo = false;
        }
        if (!wait_or_flag(&bar_pready[k & 1], (k >> 1) & 1, p, aborted)) break;
        issue_pv(k, cur.first);
        pv_todo = false;
        if (qk_todo || pv_todo || !has_next) break;
        cur = nxt;
        has_next = nxt.next();
      }
    }
    // The other groups are done with tensor memory, and every MMA has completed: in a normal
    // run the softmax group waited for each segment's last P.V; after an abort the last
    // commit is waited for here (MMAs complete on their own).  Then release tensor memory
    // (the allocating warp).
    named_sync(kBarAll, kTokThreads + 32);
    if (last_bar) mbar_wait(last_bar, last_par, p.timeout_ns);
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
    return;
  }

  const int q4 = warp & 3;
  const int t = q4 * 32 + lane;  // token of the tile = tensor-memory lane
  const uint32_t t_lane = tmem + ((uint32_t)(q4 * 32) << 16);

  if (warp >= kDqWarp0) {
    // ======================= dequant group (warps 6..17) ========================
    // Iteration k: K tile k+1 -> tensor memory.  Warp (q4, part) owns tokens 32*q4.. and
    // K blocks 6*part .. 6*part+5.
    const int dwarp = warp - kDqWarp0;  // 0..11
    const int part = dwarp >> 2;
    const int gtid = tid - kDqWarp0 * 32;  // 0..383
    // Segment j's score factors go to slot j % 4 of the ring, read by the softmax of its
    // tiles; slot j % 4 was last read by segment j - 4, whose tiles precede tile k - 2 when
    // segment j starts at tile k + 1, and the softmax group finished them before it signalled
    // tile k - 1 (waited for below).
    float* chs = reinterpret_cast<float*>(smem + kOffCh);
    // prologue: tile 0 (a segment start)
    if (gtid < kHeads) chs[(it.seg & 3) * kHeads + gtid] = p.ws.qch[it.b * kHeads + gtid];
    // a stage is converted once it landed and the reference warp wrote its reference exponent
    wait_or_flag(&bar_full[0], 0, p, aborted);
    wait_or_flag(&bar_tready[0], 0, p, aborted);
    k_tile_to_tmem(smem + kOffStages, it.n, t, part, t_lane + kColA, t_lane + kColSt,
                   *reinterpret_cast<const int*>(smem + kOffStages + kStageRefOff));
    tc_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&bar_kready[0]);
      mbar_arrive(&bar_empty[0]);
    }
    for (int k = 0; it.next(); ++k) {  // it: tile k+1
      // ---- K tile k+1 -> tensor-memory buffer (k+1)&1.  The buffer held tile k-1, read by its
      // QK^T and by the softmax group's V^T copy; both are done once the softmax group signalled
      // tile k-1 (it waited for that QK^T first) ----
      const int s1 = (k + 1) % kStages;
      const bool new_seg = it.first && gtid < kHeads;
      const float chv = new_seg ? p.ws.qch[it.b * kHeads + gtid] : 0.f;
      wait_or_flag(&bar_full[s1], ((k + 1) / kStages) & 1, p, aborted);
      wait_or_flag(&bar_tready[s1], ((k + 1) / kStages) & 1, p, aborted);
      if (k >= 1) wait_or_flag(&bar_pready[(k - 1) & 1], ((k - 1) >> 1) & 1, p, aborted);
      if (new_seg) chs[(it.seg & 3) * kHeads + gtid] = chv;
      tc_fence_after();
      // the reference of tile k+1 goes to column (k+1) % 4, last read by the softmax of tile k-3
      const uint8_t* st = smem + kOffStages + s1 * kStageBytes;
      k_tile_to_tmem(st, it.n, t, part, t_lane + kColA + kColsA * ((k + 1) & 1), t_lane + kColSt + ((k + 1) & 3),
                     *reinterpret_cast<const int*>(st + kStageRefOff));
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar_kready[(k + 1) & 1]);
        mbar_arrive(&bar_empty[s1]);
      }
    }
  } else {
    // ======================= softmax group (warps 2..5) =========================
    // Warp q4 owns tokens 32*q4.. of each tile and all 16 heads; lane L keeps the
    // running statistics of head L >> 1 (in shared memory, shared by the lane pair).
    const int sw = warp - kSmWarp0;  // 0..3
    const int stid = tid - kSmWarp0 * 32;  // 0..127
    const float* chs = reinterpret_cast<const float*>(smem + kOffCh);
    float* mstate = reinterpret_cast<float*>(smem + kOffMst) + sw * 2 * kHeads;  // [16] m, [16] alpha*resc
    float l_part[16];
    int R = 0;
    int k = 0;
    bool has_next;
    do {
      const bool valid = t < it.n;
      const bool seg_first = it.first;
      const float* ch = chs + (it.seg & 3) * kHeads;
      // S^T and the tile's reference exponent R_k (stored by the dequant group before the K
      // tile that QK^T read was declared ready; the same value in every lane)
      wait_or_flag(&bar_qk[k & 1], (k >> 1) & 1, p, aborted);
      // The P^T buffer written below (k & 1) was last read by P.V of tile k-2, which the MMA
      // warp issued before QK^T of tile k: the commit that signalled S^T of tile k covers it.
      tc_fence_after();
      int Rk;
      float s2[16];
      float* hmax = reinterpret_cast<float*>(smem + kOffHmax) + (k & 1) * 4 * kHeads;  // [16 heads][4 quarters]
      {
        uint32_t rh[16], rl[16], sv[1];
        const uint32_t scol = t_lane + kColS + 32 * (k & 1);
        tmem_ld16_nowait(scol, rh);
        tmem_ld16_nowait(scol + 16, rl);
        tmem_ld1_nowait(t_lane + kColSt + (k & 3), sv);
        tc_wait_ld();
        Rk = (int)sv[0];
        // 2^(R_k - 127 - kHead): a power of two (also where it is subnormal), so the products
        // below round only once; a tile holding a NaN scale byte (R_k = 255) gives NaN scores
        const float stok = Rk == 255 ? __int_as_float(0x7FC00000) : exp2i(Rk - 127 - kHead);
        // s = (hi + lo part scores) * (head factor * tile factor); -inf past the tile's tokens
        // (their K rows are zero)
        const float2 st2 = make_float2(stok, stok);
        const float pen = valid ? 0.f : -INFINITY;
        const float2 pen2 = make_float2(pen, pen);
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const float4 c4 = *reinterpret_cast<const float4*>(ch + i);
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            const float2 cs = f2mul(u == 0 ? make_float2(c4.x, c4.y) : make_float2(c4.z, c4.w), st2);
            const float2 sum = f2add(make_float2(__uint_as_float(rh[i + u]), __uint_as_float(rh[i + u + 1])),
                                     make_float2(__uint_as_float(rl[i + u]), __uint_as_float(rl[i + u + 1])));
            const float2 sv2 = f2fma(sum, cs, pen2);
            s2[i + u] = sv2.x;
            s2[i + u + 1] = sv2.y;
          }
        }
      }
      // d = s - m with the running maxima as they stand.  When every score of the tile is
      // within kMaxThresh of its head's maximum (one AND-reducing barrier over the group) and
      // the tile's reference equals the previous one, nothing moves: no tile maxima are
      // exchanged and P uses d as it is.  A moving maximum, a new reference or a segment
      // start takes the full path (the same decisions either way).
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
      const int Rnew = Rk;
      const bool fits = !seg_first && dmax <= (float)(kMaxThresh + kPExp) && Rnew == R;
      bool resc = false;
      if (!named_sync_and(kBarSm, kSmThreads, fits)) {
        // tile maxima: per head over the warp's tokens, then over the four warps
        const float wm = warp_reduce16<true>(s2, lane);
        if ((lane & 1) == 0) hmax[(lane >> 1) * 4 + q4] = wm;
        named_sync(kBarSm, kSmThreads);
        // running statistics: lane L computes head L >> 1; the lane pair agrees
        {
          const int h = lane >> 1;
          const float4 hm = *reinterpret_cast<const float4*>(hmax + h * 4);
          const float M = fmaxf(fmaxf(hm.x, hm.y), fmaxf(hm.z, hm.w));
          const float mo = mstate[h];
          float mn = mo, alpha = 1.f;
          bool moved = false;
          // mstate holds m - kPExp (see kPExp)
          if (seg_first) {
            mn = M - (float)kPExp;
            alpha = 0.f;
          } else if (M > mo + (float)(kPExp + kMaxThresh)) {
            mn = M - (float)kPExp;
            alpha = ex2(mo - mn);
            moved = true;
          }
          resc = __any_sync(0xffffffffu, moved) || (!seg_first && Rnew != R);
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
        // P' = hi + lo, both e5m2 (see kPExp); P' - hi is exact in f16
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
      // ---- P.V of tile k-1 must be complete: O^T rescale and V^T below ----
      if (k > 0) wait_or_flag(&bar_pv[(k - 1) & 1], ((k - 1) >> 1) & 1, p, aborted);
      tc_fence_after();
      if (resc) rescale_o(t_lane, mstate + kHeads, exp2i(R - Rnew));
      R = Rnew;
      // ---- V^T of tile k: this thread's token, all 512 dims, from the K tile in tensor memory ----
      {
        const uint32_t acol = t_lane + kColA + kColsA * (k & 1);
        uint8_t* vrow = smem + kOffVt + (t >> 3) * kVtLbo + (t & 7) * 16;
#pragma unroll 1
        for (int b4 = 0; b4 < kDv / 32; b4 += 4) {  // blocks b4 .. b4+3 = dims 32*b4 .. 32*b4+127
          uint32_t e[4][8];
#pragma unroll
          for (int j = 0; j < 4; ++j) tmem_ld8_nowait(acol + 8 * (b4 + j), e[j]);
          tc_wait_ld();
          uint8_t* d = vrow + (b4 >> 2) * kVtBlock;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            *reinterpret_cast<uint4*>(d + 2 * j * kVtSbo) = make_uint4(e[j][0], e[j][1], e[j][2], e[j][3]);
            *reinterpret_cast<uint4*>(d + (2 * j + 1) * kVtSbo) = make_uint4(e[j][4], e[j][5], e[j][6], e[j][7]);
          }
        }
      }
      fence_proxy_async_smem();  // P^T and V^T are read by the tensor cores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pready[k & 1]);
      if (it.last) {
        // ---- segment epilogue: l over the segment, then O = (hi + lo) * 2^-kHead * 2^(R-127) / l ----
        float* lw = reinterpret_cast<float*>(smem + kOffLw);      // [16 heads][4 quarters]
        float* ofac = reinterpret_cast<float*>(smem + kOffMlast);  // [16] 2^(R-127) / l
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
          const float os = (R == 255) ? __int_as_float(0x7FC00000) : exp2i(R - 127);
          ofac[h] = os / L;
        }
        named_sync(kBarSm, kSmThreads);
        wait_or_flag(&bar_pv[k & 1], (k >> 1) & 1, p, aborted);
        tc_fence_after();
        segment_out(whole ? (void*)(p.out + (long long)it.b * kHeads * kDv)
                          : (void*)(p.ws.part_acc + (long long)slot * kHeads * kDv),
                    whole, ofac, t_lane, t);
        tc_fence_before();
        named_sync(kBarSm, kSmThreads);  // lw, ofac and the accumulator are reused by the next segment
      }
      has_next = it.next();
      ++k;
    } while (has_next);
  }
  // tensor memory is released by the MMA warp once every group is past this point
  tc_fence_before();
  named_sync(kBarAll, kTokThreads + 32);
}

// ---- merge of split sequences -------------------------------------------------------
// CTA (b, y) merges heads 4y..4y+3 of sequence b (four CTAs per sequence spread the partial
// loads over more SMs), warp w = head 4y + w, lane l = dims 16l..16l+15:
// out = sum_s 2^(lse_s - M) acc_s / sum_s 2^(lse_s - M), M = max_s lse_s; empty -> zeros.
constexpr int kMergeHeads = 4;  // heads per CTA: kHeads / kMergeHeads CTAs per sequence
constexpr int kMergeThreads = 32 * kMergeHeads;
__global__ void __launch_bounds__(kMergeThreads) mla_merge_kernel(__nv_bfloat16* __restrict__ out, Workspace ws,
                                                                  int B) {
  // The partition written by the partition kernel (complete before the split kernel, this
  // grid's predecessor, started) is read while the split kernel drains; its partials only
  // after griddepcontrol.wait.
  const int b = blockIdx.x;
  const int tid = threadIdx.x, h = (tid >> 5) + kMergeHeads * blockIdx.y, lane = tid & 31;
  const int a0 = ws.ipc[b], a1 = ws.ipc[b + 1];
  uint4* dst = reinterpret_cast<uint4*>(out + ((long long)b * kHeads + h) * kDv + lane * 16);
  int f = 0, ns = 0, shift0 = 0;
  if (a1 <= a0) {  // empty sequence -> zeros (the split kernel writes no row of it)
    dst[0] = make_uint4(0, 0, 0, 0);
    dst[1] = make_uint4(0, 0, 0, 0);
  } else {
    // ranges f .. f + ns - 1 hold the sequence's tiles tp[b] .. tp[b+1] - 1 (range g holds tiles
    // from floor(g T / geff)); ns == 1: a whole sequence, written by the split kernel
    const long long T = ws.meta[kMetaTiles], geff = ws.meta[kMetaGeff];
    const int t0 = ws.tp[b], t1 = ws.tp[b + 1];
    f = (int)(((t0 + 1) * geff - 1) / T);
    ns = (int)((t1 * geff - 1) / T) - f + 1;
    shift0 = (int)(f * T / geff) != t0 ? 1 : 0;
  }
  // Every CTA waits for the split grid, also those with nothing to merge: this grid must not
  // complete before its predecessor, since the next kernel in the stream (launched
  // programmatically) may start as soon as it does and rewrites the workspace.
  grid_dependency_wait();  // the split kernel's partials
  grid_launch_dependents();  // the next call's partition kernel waits for this grid itself
  if (ns < 2) return;
  // partial i of this sequence is in slot 2(f + i), the first one shifted by one when the
  // sequence is not the first of range f
  auto slot_of = [&](int i) { return 2 * (f + i) + (i == 0 ? shift0 : 0); };
  // the rows of up to kPre partials are requested together with the weights (one round
  // trip to memory for splits of up to kPre ways)
  constexpr int kPre = 4;
  auto row = [&](int i) {
    return reinterpret_cast<const float4*>(ws.part_acc + ((long long)slot_of(i) * kHeads + h) * kDv + lane * 16);
  };
  float4 y[kPre][4];
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    const float4* pj = row(j < ns ? j : 0);
#pragma unroll
    for (int q = 0; q < 4; ++q) y[j][q] = j < ns ? pj[q] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // lane i holds the weight of partials i, i+32, ...; M over all partials first
  float M = -INFINITY;
  for (int i = lane; i < ns; i += 32) M = fmaxf(M, ws.part_lse[slot_of(i) * kHeads + h]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.f;
  auto add2 = [&](float w0, const float4 (&x0)[4], float w1, const float4 (&x1)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[4 * q] += w0 * x0[q].x + w1 * x1[q].x;
      acc[4 * q + 1] += w0 * x0[q].y + w1 * x1[q].y;
      acc[4 * q + 2] += w0 * x0[q].z + w1 * x1[q].z;
      acc[4 * q + 3] += w0 * x0[q].w + w1 * x1[q].w;
    }
  };
  auto add1 = [&](float w0, const float4 (&x0)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[4 * q] += w0 * x0[q].x;
      acc[4 * q + 1] += w0 * x0[q].y;
      acc[4 * q + 2] += w0 * x0[q].z;
      acc[4 * q + 3] += w0 * x0[q].w;
    }
  };
  float L = 0.f;
  for (int c0 = 0; c0 < ns; c0 += 32) {
    const int cn = min(32, ns - c0);
    const float wl = lane < cn ? ex2(ws.part_lse[slot_of(c0 + lane) * kHeads + h] - M) : 0.f;
    L += wl;
    int i = 0;
    if (c0 == 0) {  // the preloaded partials, in pairs (static indices into y)
#pragma unroll
      for (int pr = 0; pr < kPre; pr += 2) {
        if (i == pr && pr + 1 < cn) {
          add2(__shfl_sync(0xffffffffu, wl, pr), y[pr], __shfl_sync(0xffffffffu, wl, pr + 1), y[pr + 1]);
          i = pr + 2;
        } else if (i == pr && pr < cn) {
          add1(__shfl_sync(0xffffffffu, wl, pr), y[pr]);
          i = pr + 1;
        }
      }
    }
    for (; i + 1 < cn; i += 2) {  // two partials' loads in flight
      const float4* s0 = row(c0 + i);
      const float4* s1 = row(c0 + i + 1);
      float4 x0[4], x1[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        x0[q] = s0[q];
        x1[q] = s1[q];
      }
      add2(__shfl_sync(0xffffffffu, wl, i), x0, __shfl_sync(0xffffffffu, wl, i + 1), x1);
    }
    if (i < cn) {
      const float4* s0 = row(c0 + i);
      float4 x0[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) x0[q] = s0[q];
      add1(__shfl_sync(0xffffffffu, wl, i), x0);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = 1.f / L;
  uint32_t pk[8];
#pragma unroll
  for (int q2 = 0; q2 < 8; ++q2) {
    __nv_bfloat162 bv = __floats2bfloat162_rn(acc[2 * q2] * inv, acc[2 * q2 + 1] * inv);
    pk[q2] = *reinterpret_cast<uint32_t*>(&bv);
  }
  dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
}

}  // namespace mla
