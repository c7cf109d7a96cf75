// C ABI of libmla_mxfp4.so (declared in include/mla_mxfp4.h): host-side
// argument checks, workspace layout, per-device workspace cache, and the launch
// sequence partition -> split -> merge on one stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "mla_fp8_kernel.cuh"
#include "mla_kernels.cuh"
#include "mla_mxfp4.h"

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool init = false;
  int sms = 0;
  int grid = 0;      // resident CTAs of the MXFP4 split kernel
  int grid_fp8 = 0;  // resident CTAs of the fp8 split kernel
  int ws_grid = 0;   // the larger: workspaces are sized for either kernel
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
void* g_ws[kMaxDevices] = {};
size_t g_ws_bytes[kMaxDevices] = {};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsOffsets {
  size_t meta, ipc, cta_desc, lse, acc, qhat, qch, kvc, qoc, phys, tp, total;
};

WsOffsets ws_offsets(int batch, int grid) {
  WsOffsets o;
  size_t off = 0;
  o.meta = off;
  off = align_up(off + 16 * sizeof(int), 256);
  o.ipc = off;
  off = align_up(off + (size_t)(batch + 1) * sizeof(int), 256);
  o.cta_desc = off;
  off = align_up(off + 2 * (size_t)grid * sizeof(int4), 256);
  const size_t slots = 2 * (size_t)grid;  // split sequences need at most 2 partials per range
  o.lse = off;
  off = align_up(off + slots * mla::kHeads * sizeof(float), 256);
  o.acc = off;
  off = align_up(off + slots * mla::kHeads * mla::kDv * sizeof(float), 256);
  o.qhat = off;
  off = align_up(off + (size_t)batch * mla::kQhatBytes, 256);
  o.qch = off;
  off = align_up(off + (size_t)batch * mla::kHeads * sizeof(float), 256);
  // general layouts (several query rows per sequence, paged KV): batch counts the larger of
  // the sequences and the query rows
  o.kvc = off;
  off = align_up(off + (size_t)(batch + 1) * sizeof(int), 256);
  o.qoc = off;
  off = align_up(off + (size_t)(batch + 1) * sizeof(int), 256);
  o.phys = off;
  off = align_up(off + (size_t)batch * sizeof(int), 256);
  o.tp = off;
  off = align_up(off + (size_t)(batch + 1) * sizeof(int), 256);
  o.total = off;
  return o;
}

mla::Workspace ws_bind(void* base, const WsOffsets& o) {
  uint8_t* b = static_cast<uint8_t*>(base);
  mla::Workspace w;
  w.meta = reinterpret_cast<int*>(b + o.meta);
  w.ipc = reinterpret_cast<int*>(b + o.ipc);
  w.cta_desc = reinterpret_cast<int4*>(b + o.cta_desc);
  w.part_lse = reinterpret_cast<float*>(b + o.lse);
  w.part_acc = reinterpret_cast<float*>(b + o.acc);
  w.qhat = b + o.qhat;
  w.qch = reinterpret_cast<float*>(b + o.qch);
  w.kvc = reinterpret_cast<int*>(b + o.kvc);
  w.qoc = reinterpret_cast<int*>(b + o.qoc);
  w.phys = reinterpret_cast<int*>(b + o.phys);
  w.tp = reinterpret_cast<int*>(b + o.tp);
  return w;
}

// Called with g_mu held.
int device_info(int dev, DeviceInfo* out) {
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_ERR_CUDA;
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) return MLA_ERR_CUDA;
    int occ = 0, occ8 = 0;
    cudaError_t e = cudaFuncSetAttribute(mla::mla_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         mla::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, mla::mla_split_kernel, mla::kThreads,
                                                        mla::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mla::fp8::mla_split_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               mla::fp8::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ8, mla::fp8::mla_split_fp8_kernel, mla::fp8::kThreads,
                                                        mla::fp8::kSmemBytes);
    if (prev != dev && prev >= 0) cudaSetDevice(prev);
    if (e != cudaSuccess || occ < 1 || occ8 < 1) return MLA_ERR_CUDA;
    d.sms = sms;
    // the partition kernel cuts ranges for at most kPartMaxGrid CTAs
    d.grid = sms * occ < mla::kPartMaxGrid ? sms * occ : mla::kPartMaxGrid;
    d.grid_fp8 = sms * occ8 < mla::kPartMaxGrid ? sms * occ8 : mla::kPartMaxGrid;
    d.ws_grid = d.grid > d.grid_fp8 ? d.grid : d.grid_fp8;
    d.init = true;
  }
  *out = d;
  return MLA_OK;
}

int check_args(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale, const int32_t* kv_indptr,
               const void* out, int batch, float sm_scale) {
  if (batch < 0) return MLA_ERR_BAD_BATCH;
  if (batch == 0) return MLA_OK;
  if (!q || !kv_indptr || !out) return MLA_ERR_NULL_PTR;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv_packed) |
       reinterpret_cast<uintptr_t>(out)) & 15u)
    return MLA_ERR_BAD_ALIGN;
  if (reinterpret_cast<uintptr_t>(kv_indptr) & 3u) return MLA_ERR_BAD_ALIGN;
  if (!std::isfinite(sm_scale)) return MLA_ERR_BAD_SCALE;
  return MLA_OK;
}

// Wait limit of the split kernel's mbarrier waits (global time); a wait that runs out
// raises MLA_DEVICE_TIMEOUT and the launch returns instead of blocking.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

struct LaunchOpts {
  cudaEvent_t ev_begin = nullptr;  // recorded right before the split kernel
  cudaEvent_t ev_end = nullptr;    // recorded right after it
  unsigned long long timeout_ns = kWaitLimitNs;
  int stall_producer = 0;          // test hook (mla_decode_mxfp4_ws_stalled)
  mla::RowMap rm = {};             // general layouts (null pointers: the plain one)
  int ws_rows = -1;                // workspace sized for this many rows (default: batch)
  const CUtensorMap* fp8_map = nullptr;  // set: the fp8 kernel on this tensor map
  const float* fp8_scale = nullptr;      // its per-tensor scale (device)
};

int launch(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale, const int32_t* kv_indptr, void* out,
           int batch, float sm_scale, cudaStream_t stream, void* ws, const DeviceInfo& di,
           const LaunchOpts& opt = LaunchOpts()) {
  const cudaEvent_t ev_begin = opt.ev_begin, ev_end = opt.ev_end;
  const WsOffsets o = ws_offsets(opt.ws_rows >= 0 ? opt.ws_rows : batch, di.ws_grid);
  const int grid = opt.fp8_map ? di.grid_fp8 : di.grid;
  const mla::Workspace w = ws_bind(ws, o);
  const int kv_null = (kv_packed == nullptr || kv_scale == nullptr) ? 1 : 0;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  {
    // may be scheduled while the preceding kernel (e.g. the previous call's merge) drains;
    // it waits for that grid before its first load
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1 + (batch + mla::kQhatSeqsPerBlock - 1) / mla::kQhatSeqsPerBlock);
    cfg.blockDim = dim3(mla::kPartThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    const int tile = opt.fp8_map ? mla::fp8::kTile : mla::kTile;  // the split kernel's tile
    if (cudaLaunchKernelEx(&cfg, mla::mla_partition_kernel, kv_indptr, batch, grid, kv_null, w,
                           static_cast<const __nv_bfloat16*>(q), sm_scale, opt.rm, tile) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  mla::SplitParams sp;
  sp.kv = kv_packed;
  // kv_scale has no alignment rule: the kernel addresses it from the 16-byte boundary below it
  sp.sc_mis = (int)(reinterpret_cast<uintptr_t>(kv_scale) & 15u);
  sp.sc = reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(kv_scale) - (uintptr_t)sp.sc_mis);
  sp.out = static_cast<__nv_bfloat16*>(out);
  sp.ws = w;
  sp.B = batch;
  sp.timeout_ns = opt.timeout_ns;
  sp.stall_producer = opt.stall_producer;
  sp.rmode = opt.rm.kv_indices ? mla::kRowModePaged : (opt.rm.qo_indptr ? mla::kRowModeContig : mla::kRowModePlain);
  sp.kv_indices = opt.rm.kv_indices;
  sp.page_size = opt.rm.page_size;
  sp.num_pages = opt.rm.num_pages;
  // split and merge are launched with programmatic stream serialization: each may be
  // scheduled while its predecessor runs and waits for it with griddepcontrol.wait.  The
  // timed variant records events between the launches, which orders them as usual.
  if (ev_begin && cudaEventRecord(ev_begin, stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (opt.fp8_map) {
    mla::fp8::Fp8Params fp;
    fp.kv_scale = opt.fp8_scale;
    fp.out = static_cast<__nv_bfloat16*>(out);
    fp.ws = w;
    fp.B = batch;
    fp.rmode = opt.rm.qo_indptr ? mla::kRowModeContig : mla::kRowModePlain;
    fp.timeout_ns = opt.timeout_ns;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(mla::fp8::kThreads);
    cfg.dynamicSmemBytes = mla::fp8::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, mla::fp8::mla_split_fp8_kernel, *opt.fp8_map, fp) != cudaSuccess)
      return MLA_ERR_CUDA;
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(mla::kThreads);
    cfg.dynamicSmemBytes = mla::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, mla::mla_split_kernel, sp) != cudaSuccess) return MLA_ERR_CUDA;
  }
  if (ev_end && cudaEventRecord(ev_end, stream) != cudaSuccess) return MLA_ERR_CUDA;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(batch, mla::kHeads / mla::kMergeHeads);
    cfg.blockDim = dim3(mla::kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, mla::mla_merge_kernel, static_cast<__nv_bfloat16*>(out), w, batch) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  // every launch and event record above was checked; an error left pending on this thread
  // by unrelated work is not this call's and is left for its owner to read
  return MLA_OK;
}

// ---- static scratch for callers that cannot allocate device memory ----------
// Sized for at most kStaticMaxBatch sequences and kStaticMaxGrid resident
// split-kernel CTAs (GB300: 152), i.e. the workspace layout of ws_offsets().
constexpr int kStaticMaxBatch = 4096;
constexpr int kStaticMaxGrid = 160;
constexpr size_t static_align(size_t x) { return (x + 255) / 256 * 256; }
constexpr size_t kStaticScratchBytes =
    static_align(16 * sizeof(int)) + static_align((size_t)(kStaticMaxBatch + 1) * sizeof(int)) +
    static_align(2 * (size_t)kStaticMaxGrid * sizeof(int4)) +
    static_align(2 * (size_t)kStaticMaxGrid * mla::kHeads * sizeof(float)) +
    static_align(2 * (size_t)kStaticMaxGrid * mla::kHeads * mla::kDv * sizeof(float)) +
    static_align((size_t)kStaticMaxBatch * mla::kQhatBytes) +
    static_align((size_t)kStaticMaxBatch * mla::kHeads * sizeof(float)) +
    2 * static_align((size_t)(kStaticMaxBatch + 1) * sizeof(int)) + static_align((size_t)kStaticMaxBatch * sizeof(int)) +
    static_align((size_t)(kStaticMaxBatch + 1) * sizeof(int));

// One copy per GPU that loads the library, alive until the process exits.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch per device (host code cannot use the
// symbol's name as an address).  Filled on the first no-alloc call per device.
void* g_static_ptr[kMaxDevices] = {};

}  // namespace

namespace {
// cuTensorMapEncodeTiled from the driver, looked up once (the runtime hands out driver entry
// points, so the library links no driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Tensor map of an fp8 KV buffer [rows][576] for the fp8 kernel: boxes of 128 rows x 128 bytes
// with the 128-byte swizzle; reads past the buffer's rows or past a row's 576 bytes give zeros.
int fp8_tensor_map(const uint8_t* kv, int rows, CUtensorMap* m) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return MLA_ERR_CUDA;
  const cuuint64_t dims[2] = {(cuuint64_t)mla::kDqk, (cuuint64_t)(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {(cuuint64_t)mla::kDqk};
  const cuuint32_t box[2] = {(cuuint32_t)mla::fp8::kBoxBytes, (cuuint32_t)mla::fp8::kTile};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(kv), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

int launch_ws(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale, const int32_t* kv_indptr, void* out,
              int batch, float sm_scale, mla_stream_t stream, void* workspace, size_t ws_bytes,
              const LaunchOpts& opt) {
  int rc = check_args(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale);
  if (rc != MLA_OK || batch == 0) return rc;
  if (!workspace) return MLA_ERR_NULL_PTR;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MLA_ERR_BAD_ALIGN;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  DeviceInfo di;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    rc = device_info(dev, &di);
  }
  if (rc != MLA_OK) return rc;
  if (ws_bytes < ws_offsets(opt.ws_rows >= 0 ? opt.ws_rows : batch, di.ws_grid).total) return MLA_ERR_WORKSPACE;
  return launch(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale, reinterpret_cast<cudaStream_t>(stream),
                workspace, di, opt);
}
}  // namespace

extern "C" {

size_t mla_decode_mxfp4_workspace_bytes(int batch, int device) {
  if (batch < 0) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo di;
  if (device_info(device, &di) != MLA_OK) return 0;
  return ws_offsets(batch, di.ws_grid).total;
}


int mla_decode_mxfp4_ws_timed(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                              const int32_t* kv_indptr, void* out, int batch, float sm_scale, mla_stream_t stream,
                              void* workspace, size_t ws_bytes, void* ev_split_begin, void* ev_split_end) {
  LaunchOpts opt;
  opt.ev_begin = static_cast<cudaEvent_t>(ev_split_begin);
  opt.ev_end = static_cast<cudaEvent_t>(ev_split_end);
  return launch_ws(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale, stream, workspace, ws_bytes, opt);
}

int mla_decode_mxfp4_ws_stalled(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                                const int32_t* kv_indptr, void* out, int batch, float sm_scale,
                                mla_stream_t stream, void* workspace, size_t ws_bytes,
                                unsigned long long timeout_ns) {
  if (timeout_ns == 0 || timeout_ns > kWaitLimitNs) return MLA_ERR_BAD_SCALE;
  LaunchOpts opt;
  opt.timeout_ns = timeout_ns;
  opt.stall_producer = 1;
  return launch_ws(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale, stream, workspace, ws_bytes, opt);
}

int mla_decode_mxfp4_paged_ws_timed(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                                    const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
                                    const int32_t* kv_last_page_len, int page_size, int num_pages, void* out,
                                    int batch, int total_q, float sm_scale, mla_stream_t stream, void* workspace,
                                    size_t ws_bytes, void* ev_split_begin, void* ev_split_end) {
  if (batch < 0 || total_q < 0) return MLA_ERR_BAD_BATCH;
  if (!qo_indptr && total_q != batch) return MLA_ERR_BAD_LAYOUT;
  if (kv_indices) {
    if (page_size < 1 || num_pages < 0 || !kv_last_page_len) return MLA_ERR_BAD_LAYOUT;
    if (reinterpret_cast<uintptr_t>(kv_indices) & 3u) return MLA_ERR_BAD_ALIGN;
    if (reinterpret_cast<uintptr_t>(kv_last_page_len) & 3u) return MLA_ERR_BAD_ALIGN;
  }
  if (qo_indptr && (reinterpret_cast<uintptr_t>(qo_indptr) & 3u)) return MLA_ERR_BAD_ALIGN;
  if (total_q == 0) return MLA_OK;
  if (batch == 0) {
    // query rows but no sequence: every row is empty (zeros), like an empty sequence
    if (!out) return MLA_ERR_NULL_PTR;
    if (reinterpret_cast<uintptr_t>(out) & 15u) return MLA_ERR_BAD_ALIGN;
    return cudaMemsetAsync(out, 0, (size_t)total_q * mla::kHeads * mla::kDv * 2, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
  }
  LaunchOpts opt;
  opt.ev_begin = static_cast<cudaEvent_t>(ev_split_begin);
  opt.ev_end = static_cast<cudaEvent_t>(ev_split_end);
  opt.rm.qo_indptr = qo_indptr;
  opt.rm.kv_indices = kv_indices;
  opt.rm.last_len = kv_last_page_len;
  opt.rm.Bkv = batch;
  opt.rm.page_size = kv_indices ? page_size : 0;
  opt.rm.num_pages = kv_indices ? num_pages : 0;
  opt.ws_rows = batch > total_q ? batch : total_q;
  // the kernels run over the query rows; with neither map this is the plain decode
  return launch_ws(q, kv_packed, kv_scale, kv_indptr, out, total_q, sm_scale, stream, workspace, ws_bytes, opt);
}

int mla_decode_mxfp4_paged_ws(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                              const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
                              const int32_t* kv_last_page_len, int page_size, int num_pages, void* out, int batch,
                              int total_q, float sm_scale, mla_stream_t stream, void* workspace, size_t ws_bytes) {
  return mla_decode_mxfp4_paged_ws_timed(q, kv_packed, kv_scale, qo_indptr, kv_indptr, kv_indices, kv_last_page_len,
                                         page_size, num_pages, out, batch, total_q, sm_scale, stream, workspace,
                                         ws_bytes, nullptr, nullptr);
}

int mla_decode_fp8_ws_timed(const void* q, const uint8_t* kv_fp8, const float* kv_scale, const int32_t* qo_indptr,
                            const int32_t* kv_indptr, int kv_rows, void* out, int batch, int total_q, float sm_scale,
                            mla_stream_t stream, void* workspace, size_t ws_bytes, void* ev_split_begin,
                            void* ev_split_end) {
  if (batch < 0 || total_q < 0 || kv_rows < 0) return MLA_ERR_BAD_BATCH;
  if (!qo_indptr && total_q != batch) return MLA_ERR_BAD_LAYOUT;
  if (qo_indptr && (reinterpret_cast<uintptr_t>(qo_indptr) & 3u)) return MLA_ERR_BAD_ALIGN;
  if (total_q == 0) return MLA_OK;
  if (!kv_scale) return MLA_ERR_NULL_PTR;
  if (reinterpret_cast<uintptr_t>(kv_scale) & 3u) return MLA_ERR_BAD_ALIGN;
  if (batch == 0 || kv_rows == 0 || !kv_fp8) {
    // no KV rows: every query row is empty (zeros), as for an empty sequence
    if (!out) return MLA_ERR_NULL_PTR;
    if (reinterpret_cast<uintptr_t>(out) & 15u) return MLA_ERR_BAD_ALIGN;
    return cudaMemsetAsync(out, 0, (size_t)total_q * mla::kHeads * mla::kDv * 2,
                           reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
  }
  if (reinterpret_cast<uintptr_t>(kv_fp8) & 15u) return MLA_ERR_BAD_ALIGN;
  CUtensorMap map;
  int rc = fp8_tensor_map(kv_fp8, kv_rows, &map);
  if (rc != MLA_OK) return rc;
  LaunchOpts opt;
  opt.ev_begin = static_cast<cudaEvent_t>(ev_split_begin);
  opt.ev_end = static_cast<cudaEvent_t>(ev_split_end);
  opt.rm.qo_indptr = qo_indptr;
  opt.rm.Bkv = batch;
  opt.rm.kv_rows = kv_rows;
  opt.ws_rows = batch > total_q ? batch : total_q;
  opt.fp8_map = &map;
  opt.fp8_scale = kv_scale;
  // kv_packed = kv_fp8 (checked for alignment), kv_scale unused by this kernel (non-null marker)
  return launch_ws(q, kv_fp8, kv_fp8, kv_indptr, out, total_q, sm_scale, stream, workspace, ws_bytes, opt);
}

int mla_decode_fp8_ws(const void* q, const uint8_t* kv_fp8, const float* kv_scale, const int32_t* qo_indptr,
                      const int32_t* kv_indptr, int kv_rows, void* out, int batch, int total_q, float sm_scale,
                      mla_stream_t stream, void* workspace, size_t ws_bytes) {
  return mla_decode_fp8_ws_timed(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, kv_rows, out, batch, total_q, sm_scale,
                                 stream, workspace, ws_bytes, nullptr, nullptr);
}

int mla_decode_mxfp4_ws(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                        const int32_t* kv_indptr, void* out, int batch, float sm_scale, mla_stream_t stream,
                        void* workspace, size_t ws_bytes) {
  return launch_ws(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale, stream, workspace, ws_bytes,
                   LaunchOpts());
}

int mla_decode_mxfp4(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale, const int32_t* kv_indptr,
                     void* out, int batch, float sm_scale, mla_stream_t stream) {
  int rc = check_args(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale);
  if (rc != MLA_OK || batch == 0) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  void* ws = nullptr;
  DeviceInfo di;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    rc = device_info(dev, &di);
    if (rc != MLA_OK) return rc;
    const size_t need = ws_offsets(batch, di.ws_grid).total;
    if (g_ws_bytes[dev] < need) {
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cs) != cudaSuccess) return MLA_ERR_CUDA;
      if (cs != cudaStreamCaptureStatusNone) return MLA_ERR_WORKSPACE;
      if (g_ws[dev]) {
        cudaDeviceSynchronize();
        cudaFree(g_ws[dev]);
        g_ws[dev] = nullptr;
        g_ws_bytes[dev] = 0;
      }
      const size_t grow = need + need / 4;
      if (cudaMalloc(&g_ws[dev], grow) != cudaSuccess) {
        g_ws[dev] = nullptr;
        return MLA_ERR_CUDA;
      }
      g_ws_bytes[dev] = grow;
    }
    ws = g_ws[dev];
  }
  return launch(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale, reinterpret_cast<cudaStream_t>(stream), ws,
                di);
}

int mla_decode_mxfp4_noalloc(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                             const int32_t* kv_indptr, void* out, int batch, float sm_scale,
                             mla_stream_t stream) {
  int rc = check_args(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale);
  if (rc != MLA_OK || batch == 0) return rc;
  if (batch > kStaticMaxBatch) return MLA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  DeviceInfo di;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    rc = device_info(dev, &di);
    if (rc != MLA_OK) return rc;
    if (di.ws_grid > kStaticMaxGrid) return MLA_ERR_WORKSPACE;
    if (!g_static_ptr[dev]) {
      // set-up, once per device, with that device current
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return MLA_ERR_CUDA;
      g_static_ptr[dev] = ptr;
    }
    scratch = g_static_ptr[dev];
  }
  if (ws_offsets(batch, di.ws_grid).total > kStaticScratchBytes) return MLA_ERR_WORKSPACE;
  return launch(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale, reinterpret_cast<cudaStream_t>(stream),
                scratch, di);
}

int mla_decode_mxfp4_device_status(mla_stream_t stream, const void* workspace, int* status) {
  if (!status) return MLA_ERR_NULL_PTR;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  const void* ws = workspace;
  if (!ws || ws == MLA_STATIC_SCRATCH) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
    ws = ws ? g_static_ptr[dev] : g_ws[dev];
    if (!ws) {  // no call has used it on this device yet
      *status = 0;
      return MLA_OK;
    }
  }
  int meta[16];
  if (cudaMemcpy(meta, ws, sizeof(meta), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
  *status = meta[mla::kMetaStatus];
  return MLA_OK;
}

int mla_decode_mxfp4_last_device_status(mla_stream_t stream, int* status) {
  return mla_decode_mxfp4_device_status(stream, nullptr, status);
}

void mla_decode_mxfp4_release(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int prev = -1;
  cudaGetDevice(&prev);
  for (int d = 0; d < kMaxDevices; ++d) {
    if (!g_ws[d]) continue;
    cudaSetDevice(d);
    cudaDeviceSynchronize();
    cudaFree(g_ws[d]);
    g_ws[d] = nullptr;
    g_ws_bytes[d] = 0;
  }
  if (prev >= 0) cudaSetDevice(prev);
}

int mla_host_device_pointer(const void* host, void** device) {
  if (!host || !device) return MLA_ERR_NULL_PTR;
  *device = nullptr;
  // (an unregistered pointer is reported as such, not as an error, so the runtime's last-error
  // state is left as it was)
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) return MLA_ERR_CUDA;
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return MLA_ERR_CUDA;
  *device = a.devicePointer;
  return MLA_OK;
}

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_NULL_PTR: return "MLA_ERR_NULL_PTR: q, kv_indptr, out or workspace is NULL";
    case MLA_ERR_BAD_BATCH: return "MLA_ERR_BAD_BATCH: batch < 0";
    case MLA_ERR_BAD_ALIGN: return "MLA_ERR_BAD_ALIGN: misaligned pointer";
    case MLA_ERR_BAD_SCALE: return "MLA_ERR_BAD_SCALE: sm_scale is not finite";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace too small or cannot grow during capture";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: CUDA runtime error";
    case MLA_ERR_BAD_LAYOUT: return "MLA_ERR_BAD_LAYOUT: query rows or page layout arguments are inconsistent";
    default: return "unknown mla_status";
  }
}

}  // extern "C"
