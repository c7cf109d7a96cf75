/*
 * mla_mxfp4.h — C ABI of the GB300 (sm_103a) MXFP4 MLA decode-attention library
 * (libmla_mxfp4.so).
 *
 * Operation (single-token decode, DeepSeek-style absorbed multi-head latent
 * attention with one shared KV head stored as MXFP4).  Defined by the
 * kernelindex "amd-mixed-mla" submissions: tensor contract and input checks in
 * 608791 ("check_mla_inputs", "mla_decode_forward"), the MXFP4 element/scale
 * decode in 608791 (kFp4Lut, e8m0_to_float, unpack_mxfp4) and 717900
 * ("_nibble_to_f32"), the attention itself in 676098 ("_naive_fallback",
 * "_mla_fused_decode_kernel") and the split-KV log-sum-exp merge in 608791
 * ("mla_reduce_v1_like_kernel") and 676098 ("_mla_reduce_kernel"):
 *
 *   K[t][d] = e2m1(kv_packed[t][d/2] nibble) * 2^(kv_scale[t][d/32] - 127), d < 576
 *   V[t][d] = K[t][d]                                                       d < 512
 *   out[b][h][:] = sum_t softmax_t(sm_scale * q[b][h] . K[t]) V[t],
 *                  t over rows [kv_indptr[b], kv_indptr[b+1])
 *
 * Layouts (all row-major, contiguous):
 *   q          bf16  [batch][16][576]   (query row b is sequence b: one query token per sequence)
 *   kv_packed  uint8 [rows][288]        byte j = element 2j (bits 3..0) | element 2j+1 (bits 7..4)
 *   kv_scale   uint8 [rows][18]         E8M0; byte 0xFF is NaN, byte 0 is 2^-127
 *   kv_indptr  int32 [batch+1]          device memory; rows used are [kv_indptr[0], kv_indptr[batch])
 *   out        bf16  [batch][16][512]   written for every b (an empty sequence gives zeros)
 * Buffers must hold at least kv_indptr[batch] rows.  q, kv_packed and out must be
 * 16-byte aligned, kv_indptr 4-byte aligned; kv_scale has no alignment rule (bytes
 * before its first and after its last 16-byte boundary are read with plain loads).
 * out must not alias any input.  kv_packed and kv_scale may be NULL when there are
 * no KV rows; the device then treats every sequence as empty (zero output) and
 * flags MLA_DEVICE_BAD_INDPTR if kv_indptr claims rows.
 *
 * Every pointer argument is a DEVICE pointer on the current CUDA device, owned
 * by the caller.  Calls are asynchronous on `stream` (no host synchronisation,
 * no host reads of device data, no CPU fallback).  The result matches the fp64
 * definition above to |err| <= 2e-2 + 2e-2*|ref| per element (in practice far
 * tighter; see the test suite).
 *
 * Error behaviour: functions return an mla_status code.  Argument errors are
 * detected on the host before anything is launched.  A malformed kv_indptr
 * (negative entries, entries above kv_indptr[batch], or decreasing) cannot be
 * seen by the host without a synchronisation, so the device clamps it into a
 * non-decreasing sequence within [0, kv_indptr[batch]] (every access stays
 * inside the documented buffers) and raises MLA_DEVICE_BAD_INDPTR in the device
 * status word, readable with mla_decode_mxfp4_device_status().
 */
#ifndef MLA_MXFP4_H
#define MLA_MXFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle; identical to cudaStream_t (NULL = legacy default stream). */
typedef struct CUstream_st* mla_stream_t;

enum mla_status {
  MLA_OK = 0,
  MLA_ERR_NULL_PTR = 1,   /* q, kv_indptr or out is NULL (batch > 0)              */
  MLA_ERR_BAD_BATCH = 2,  /* batch < 0                                             */
  MLA_ERR_BAD_ALIGN = 3,  /* q / kv_packed / out not 16-byte, kv_indptr not 4-byte */
  MLA_ERR_BAD_SCALE = 4,  /* sm_scale is not finite                                */
  MLA_ERR_WORKSPACE = 5,  /* workspace too small, or would have to grow during
                             stream capture                                        */
  MLA_ERR_CUDA = 6,       /* a CUDA runtime call or kernel launch failed           */
  MLA_ERR_BAD_LAYOUT = 7  /* mla_decode_mxfp4_paged_ws: total_q != batch without
                             qo_indptr, page_size < 1, num_pages < 0, or
                             kv_last_page_len missing with kv_indices             */
};

/* Bits of the device status word (OR-ed; cleared at the start of every call). */
enum mla_device_status {
  MLA_DEVICE_OK = 0,
  MLA_DEVICE_BAD_INDPTR = 1, /* kv_indptr malformed (see above); clamped               */
  MLA_DEVICE_TIMEOUT = 2     /* an internal wait hit its time limit; output invalid   */
};

/*
 * Decode `batch` sequences (see top of file).  batch == 0 is a no-op returning
 * MLA_OK.  Uses a per-device workspace owned by the library, created or grown on
 * demand with cudaMalloc (which synchronises the device); it never grows while
 * `stream` is capturing (returns MLA_ERR_WORKSPACE instead), so capture a graph
 * only after one eager call of at least the same batch size, or use
 * mla_decode_mxfp4_ws.  Calls that share this workspace must be ordered (same
 * stream, or synchronised); concurrent streams should use mla_decode_mxfp4_ws.
 */
int mla_decode_mxfp4(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                     const int32_t* kv_indptr, void* out, int batch, float sm_scale,
                     mla_stream_t stream);

/* Bytes of device workspace mla_decode_mxfp4_ws needs for `batch` sequences on
 * CUDA device `device` (host-computable upper bound; 0 on error). */
size_t mla_decode_mxfp4_workspace_bytes(int batch, int device);

/* Same as mla_decode_mxfp4 but with a caller-owned device workspace of `ws_bytes`
 * bytes (at least mla_decode_mxfp4_workspace_bytes(batch, device), 256-byte
 * aligned).  Allocates nothing; safe to capture in a CUDA graph.  The workspace
 * must not be used by another call that may run concurrently. */
int mla_decode_mxfp4_ws(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                        const int32_t* kv_indptr, void* out, int batch, float sm_scale,
                        mla_stream_t stream, void* workspace, size_t ws_bytes);

/* Profiling variant of mla_decode_mxfp4_ws: additionally records `ev_split_begin`
 * and `ev_split_end` (cudaEvent_t handles, either may be NULL) on `stream`
 * immediately before and after the split-KV attention kernel, so that the
 * caller can time the dominant kernel alone with cudaEventElapsedTime.  Same
 * arguments, ownership and errors as mla_decode_mxfp4_ws. */
int mla_decode_mxfp4_ws_timed(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                              const int32_t* kv_indptr, void* out, int batch, float sm_scale,
                              mla_stream_t stream, void* workspace, size_t ws_bytes,
                              void* ev_split_begin, void* ev_split_end);

/*
 * General layouts: several query rows per sequence and/or paged KV.
 *
 * Several query rows per sequence (MTP / speculative decode; kernelindex amd-mixed-mla
 * 676098 "_naive_fallback" and 608791 "_build_decode_metadata"'s qo_indptr): with qo_indptr
 * non-NULL, query rows [qo_indptr[b], qo_indptr[b+1]) of sequence b each attend, with no
 * mask, to all of sequence b's KV rows; q is bf16 [total_q][16][576] and out bf16
 * [total_q][16][512] (a row outside every sequence's range gives zeros).  With qo_indptr
 * NULL, total_q must equal batch and row b is sequence b's single query.
 *
 * Paged KV (676098 "_aiter_mla_decode": kv_indptr over kv_indices, kv_last_page_len): with
 * kv_indices non-NULL, kv_indptr[b]..kv_indptr[b+1] index kv_indices, whose entries are page
 * ids in [0, num_pages); page p holds physical rows [p*page_size, (p+1)*page_size) of
 * kv_packed and kv_scale (so both buffers hold num_pages*page_size rows), and sequence b's
 * KV rows are, in order, its pages' rows, all page_size of them except kv_last_page_len[b]
 * (1..page_size) of its last page.  A sequence with no pages is empty.  page_size may be any
 * positive value; multiples of 8 keep the scale rows of every page 16-byte congruent, so
 * they are bulk-copied (other sizes are read with plain loads: correct, slower).  With
 * kv_indices NULL, kv_indptr counts rows as in mla_decode_mxfp4 (page_size, num_pages and
 * kv_last_page_len are ignored).
 *
 * Out-of-range page ids are clamped into the buffers and raise MLA_DEVICE_BAD_INDPTR, as do
 * malformed kv_indptr / qo_indptr (clamped to non-decreasing sequences within their ranges)
 * and kv_last_page_len outside 1..page_size (clamped).  The workspace must hold at least
 * mla_decode_mxfp4_workspace_bytes(max(batch, total_q), device) bytes, 256-byte aligned; the
 * other arguments, layouts and errors are those of mla_decode_mxfp4_ws.  The _timed variant
 * records `ev_split_begin` / `ev_split_end` (either may be NULL) around the attention kernel,
 * as mla_decode_mxfp4_ws_timed does.
 */
int mla_decode_mxfp4_paged_ws(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                              const int32_t* qo_indptr, const int32_t* kv_indptr,
                              const int32_t* kv_indices, const int32_t* kv_last_page_len,
                              int page_size, int num_pages, void* out, int batch, int total_q,
                              float sm_scale, mla_stream_t stream, void* workspace, size_t ws_bytes);
int mla_decode_mxfp4_paged_ws_timed(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                                    const int32_t* qo_indptr, const int32_t* kv_indptr,
                                    const int32_t* kv_indices, const int32_t* kv_last_page_len,
                                    int page_size, int num_pages, void* out, int batch, int total_q,
                                    float sm_scale, mla_stream_t stream, void* workspace,
                                    size_t ws_bytes, void* ev_split_begin, void* ev_split_end);

/*
 * fp8 KV with one per-tensor scale (the pages' production path: kernelindex amd-mixed-mla
 * 676098 "_aiter_mla_decode", 717900 "_decode"):
 *
 *   K[t][d] = e4m3(kv_fp8[t][d]) * (*kv_scale),  d < 576;   V[t][d] = K[t][d],  d < 512
 *   out[r][h][:] = sum_t softmax_t(sm_scale * q[r][h] . K[t]) V[t]
 *
 * over sequence b's rows [kv_indptr[b], kv_indptr[b+1]) for each of its query rows r (one per
 * sequence with qo_indptr NULL, total_q == batch; else rows [qo_indptr[b], qo_indptr[b+1]) as
 * for mla_decode_mxfp4_paged_ws).  e4m3 is the OCP "fn" encoding (no infinities; 0x7F/0xFF
 * are NaN).  The query is used as given (bf16).
 *
 * Layouts: q bf16 [total_q][16][576] (16-byte aligned); kv_fp8 uint8 [kv_rows][576] (16-byte
 * aligned; kv_rows > 0 is the number of rows the buffer holds: kv_indptr is clamped to it,
 * raising MLA_DEVICE_BAD_INDPTR, so no row outside the buffer is read); kv_scale a DEVICE
 * pointer to one float (read by the kernel, so it may change between calls, or inside a
 * captured graph, without the host reading it); kv_indptr int32 [batch+1]; out bf16
 * [total_q][16][512].  Workspace: at least mla_decode_mxfp4_workspace_bytes(max(batch,
 * total_q), device) bytes, 256-byte aligned.  Errors as mla_decode_mxfp4_paged_ws.  The _timed
 * variant records events around the attention kernel.
 */
int mla_decode_fp8_ws(const void* q, const uint8_t* kv_fp8, const float* kv_scale,
                      const int32_t* qo_indptr, const int32_t* kv_indptr, int kv_rows, void* out,
                      int batch, int total_q, float sm_scale, mla_stream_t stream, void* workspace,
                      size_t ws_bytes);
int mla_decode_fp8_ws_timed(const void* q, const uint8_t* kv_fp8, const float* kv_scale,
                            const int32_t* qo_indptr, const int32_t* kv_indptr, int kv_rows,
                            void* out, int batch, int total_q, float sm_scale, mla_stream_t stream,
                            void* workspace, size_t ws_bytes, void* ev_split_begin,
                            void* ev_split_end);

/* Test-only variant of mla_decode_mxfp4_ws that exercises the failure path of the
 * attention kernel's bounded waits without faulting anything: the kernel's copy
 * role issues no copy at all, so the first wait for a landed tile runs out after
 * `timeout_ns` nanoseconds of global time (1 .. 1e9; other values return
 * MLA_ERR_BAD_SCALE).  Every role then stops issuing asynchronous work, drains what
 * it issued and runs to its end; the call completes, `out` holds unspecified
 * values, and the workspace's device status word has MLA_DEVICE_TIMEOUT set.  The
 * context stays usable.  Same arguments, ownership and errors otherwise as
 * mla_decode_mxfp4_ws. */
int mla_decode_mxfp4_ws_stalled(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                                const int32_t* kv_indptr, void* out, int batch, float sm_scale,
                                mla_stream_t stream, void* workspace, size_t ws_bytes,
                                unsigned long long timeout_ns);

/* No-allocation variant of mla_decode_mxfp4, for callers that may not allocate
 * device memory at all: code running inside an allocator or memory-pool
 * callback, processes whose device memory is fully reserved up front by a
 * serving runtime, or hosts whose policy forbids cudaMalloc after start-up.
 * (The pages have no counterpart; this entry point is a property of this
 * library's C interface only.)
 *
 * Same arguments, layouts and results as mla_decode_mxfp4.  Instead of a
 * workspace it uses one scratch array that the library defines statically in
 * device memory: about 86 MB per GPU that loads the library, held until the
 * process exits, sized for at most 4096 sequences per call and at most 160
 * resident CTAs of the attention kernel (152 on GB300).  Larger requests are
 * rejected with MLA_ERR_WORKSPACE before anything is launched.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * The array is part of the library's device code, so it is reserved when that
 * code is loaded onto a device: under CUDA's lazy module loading that is the first
 * call of any entry point on that device.  The first call of this function on each
 * device also looks up the array's device address (cudaGetSymbolAddress) with that
 * device current.  So make one call on each device at start-up, before device
 * memory is fully reserved and before any stream capture; until then a call can
 * fail with MLA_ERR_CUDA.  Every call on a device shares the one array and it keeps
 * the previous call's contents; nothing in it needs to start at zero (each call
 * rewrites the metadata it reads), but calls that may overlap on the GPU (other
 * streams, other host threads) race on it and must be ordered by the caller.  The
 * array's device status word is read with mla_decode_mxfp4_device_status(stream,
 * MLA_STATIC_SCRATCH, &status). */
int mla_decode_mxfp4_noalloc(const void* q, const uint8_t* kv_packed, const uint8_t* kv_scale,
                             const int32_t* kv_indptr, void* out, int batch, float sm_scale,
                             mla_stream_t stream);

/* Pass as `workspace` to mla_decode_mxfp4_device_status to read the status word of
 * the static scratch array that mla_decode_mxfp4_noalloc uses. */
#define MLA_STATIC_SCRATCH ((const void*)1)

/* Debug: synchronise `stream`, then read the device status word (mla_device_status
 * bits) left by the last call that used `workspace` (NULL = the library workspace
 * of the current device, MLA_STATIC_SCRATCH = the no-allocation scratch of the
 * current device).  A workspace no call has used yet reads as 0.  Returns MLA_OK
 * or MLA_ERR_CUDA. */
int mla_decode_mxfp4_device_status(mla_stream_t stream, const void* workspace, int* status);

/* Same for the library workspace of the current device: the status of the last
 * mla_decode_mxfp4 call (equivalent to mla_decode_mxfp4_device_status(stream, NULL,
 * status)). */
int mla_decode_mxfp4_last_device_status(mla_stream_t stream, int* status);

/* Free the library-owned workspaces of every device (synchronises each device
 * that had one).  Safe to call at any time when no call is in flight. */
void mla_decode_mxfp4_release(void);

/* Device address of `host`, an address inside a page-locked host allocation that is
 * mapped into the device's address space (cudaHostAlloc, cudaHostRegister with mapping;
 * under unified addressing every page-locked allocation is), written to *device.  Passing
 * that address as q, kv_packed or kv_scale to a decode entry point makes its kernels read
 * the host buffer in place over the host link, with no copy into device memory first (the
 * inputs are read once per call; kv_indptr, out and the workspace are better kept in device
 * memory, as they are read or written many times).  The host buffer must stay allocated and
 * unmodified until the call has completed on its stream.  Returns MLA_OK, MLA_ERR_NULL_PTR, or
 * MLA_ERR_CUDA when `host` is not mapped page-locked memory (*device is then NULL). */
int mla_host_device_pointer(const void* host, void** device);

/* Human-readable name of an mla_status code. */
const char* mla_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_MXFP4_H */
