// C ABI of libmla_mxfp4.so (declared in include/mla_mxfp4.h): host-side
// argument checks, workspace layout, per-device workspace cache, and the launch
// sequence partition -> split -> merge on one stream.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "mla_kernels.cuh"
#include "mla_mxfp4.h"

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool init = false;
  int sms = 0;
  int grid = 0;  // resident CTAs of the split kernel
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
void* g_ws[kMaxDevices] = {};
size_t g_ws_bytes[kMaxDevices] = {};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsOffsets {
  size_t meta, ipc, cta_desc, lse, acc, qhat, qch, total;
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
    int occ = 0;
    cudaError_t e = cudaFuncSetAttribute(mla::mla_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         mla::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, mla::mla_split_kernel, mla::kThreads,
                                                        mla::kSmemBytes);
    if (prev != dev && prev >= 0) cudaSetDevice(prev);
    if (e != cudaSuccess || occ < 1) return MLA_ERR_CUDA;
    d.sms = sms;
    d.grid = sms * occ;
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
};

int launch(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale, const int32_t* kv_indptr, void* out,
           int batch, float sm_scale, cudaStream_t stream, void* ws, const DeviceInfo& di,
           const LaunchOpts& opt = LaunchOpts()) {
  const cudaEvent_t ev_begin = opt.ev_begin, ev_end = opt.ev_end;
  const WsOffsets o = ws_offsets(batch, di.grid);
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
    if (cudaLaunchKernelEx(&cfg, mla::mla_partition_kernel, kv_indptr, batch, di.grid, kv_null, w,
                           static_cast<const __nv_bfloat16*>(q), sm_scale) != cudaSuccess)
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
  // split and merge are launched with programmatic stream serialization: each may be
  // scheduled while its predecessor runs and waits for it with griddepcontrol.wait.  The
  // timed variant records events between the launches, which orders them as usual.
  if (ev_begin && cudaEventRecord(ev_begin, stream) != cudaSuccess) return MLA_ERR_CUDA;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(di.grid);
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
    static_align((size_t)kStaticMaxBatch * mla::kHeads * sizeof(float));

// One copy per GPU that loads the library, alive until the process exits.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch per device (host code cannot use the
// symbol's name as an address).  Filled on the first no-alloc call per device.
void* g_static_ptr[kMaxDevices] = {};

}  // namespace

namespace {
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
  if (ws_bytes < ws_offsets(batch, di.grid).total) return MLA_ERR_WORKSPACE;
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
  return ws_offsets(batch, di.grid).total;
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
    const size_t need = ws_offsets(batch, di.grid).total;
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
    if (di.grid > kStaticMaxGrid) return MLA_ERR_WORKSPACE;
    if (!g_static_ptr[dev]) {
      // set-up, once per device, with that device current
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return MLA_ERR_CUDA;
      g_static_ptr[dev] = ptr;
    }
    scratch = g_static_ptr[dev];
  }
  if (ws_offsets(batch, di.grid).total > kStaticScratchBytes) return MLA_ERR_WORKSPACE;
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

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_NULL_PTR: return "MLA_ERR_NULL_PTR: q, kv_indptr, out or workspace is NULL";
    case MLA_ERR_BAD_BATCH: return "MLA_ERR_BAD_BATCH: batch < 0";
    case MLA_ERR_BAD_ALIGN: return "MLA_ERR_BAD_ALIGN: misaligned pointer";
    case MLA_ERR_BAD_SCALE: return "MLA_ERR_BAD_SCALE: sm_scale is not finite";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace too small or cannot grow during capture";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: CUDA runtime error";
    default: return "unknown mla_status";
  }
}

}  // extern "C"
