/*
 * spconv.h -- C ABI of libspconv: forward 2-D convolution of a dense NCHW fp32
 * activation tensor with unstructured-sparse (pruned) weights, computed
 * directly on the GPU (GB300, sm_103a) without materialising an im2col matrix.
 *
 * Operation (Tuteja et al., "Theoretical and Empirical Analysis of Sparse
 * Convolution", Sec. 3 Eq.(1)-(3); Escoin, arXiv 1802.10280, "Sparse
 * convolution", Algorithm 2):
 *
 *   Y[n,m,e,f] = sum over nonzeros j of row m of value[j] *
 *                X[n, c_j, e*stride + r_j - pad, f*stride + s_j - pad]
 *
 * with X taken as zero outside [0,H) x [0,W) (symmetric zero padding, no
 * kernel flip), E = floor((H + 2*pad - R)/stride) + 1 and likewise F (Eq.(2)).
 * The weights are the M x (C*R*S) lowered filter matrix (Escoin Fig. 3) held
 * in CSR (Escoin, "Sparse weights": rowptr[M+1], colidx[nnz], value[nnz]);
 * colidx = (c*R + r)*S + s.
 *
 * Conventions shared by every call:
 *  - Return value: SPCONV_OK (0) or a negative spconv_status.  No call aborts,
 *    throws or prints; spconv_status_string() names a status.
 *  - Tensors are contiguous row-major: X is N x C x H x W, Y is N x M x E x F,
 *    both float32 in device memory of the device that was current when the
 *    handle was packed (spconv_forward_host: in host memory, with device
 *    workspaces).
 *  - "stream" is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - All shape arguments are int; sizes are validated before any device work.
 */
#ifndef SPCONV_H
#define SPCONV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum spconv_status {
    SPCONV_OK = 0,
    SPCONV_ERR_INVALID_ARG = -1, /* bad shape, NULL pointer, misaligned buffer     */
    SPCONV_ERR_BAD_CSR = -2,     /* rowptr not monotone / colidx out of range / dup */
    SPCONV_ERR_UNSUPPORTED = -3, /* shape beyond what the kernels were built for     */
    SPCONV_ERR_ALLOC = -4,       /* host or device allocation failed                 */
    SPCONV_ERR_CUDA = -5,        /* a CUDA runtime call or kernel launch failed      */
    SPCONV_ERR_MISMATCH = -6,    /* forward shape/device differs from the packed one */
    SPCONV_ERR_DEVICE = -7       /* a kernel reported a failure (see spconv_device_status) */
} spconv_status;

/* Opaque handle of a packed weight set.  Owned by the library from
 * spconv_pack / spconv_pack_host until spconv_packed_free. */
typedef struct spconv_packed spconv_packed;

/*
 * spconv_pack -- CSR -> packed device layout (once per weight set).
 *
 * Follows Escoin's "weight stretching" (the column index of every nonzero is
 * rewritten once, ahead of time, into an offset into the input array, relying
 * on the layout function f(c, y+r, x+s) = f(c,y,x) + f(0,r,s)) and the per
 * output channel offset array of Tuteja et al. Sec. 5.3.  Here each nonzero
 * becomes an 8-byte entry (fp32 value, int32 offset into the shared-memory
 * input tile the kernel stages), entries are grouped per output channel and
 * input-channel chunk, and output channels are binned by nonzero count onto
 * warps (longest-first onto the least-loaded warp).
 *
 * Inputs (host memory, caller-owned, only read during the call):
 *   C, H, W      input channels and spatial size of the layer (>= 1)
 *   M            output channels (rows of the CSR matrix, >= 1)
 *   R, S         kernel height and width (>= 1); stride >= 1; pad >= 0;
 *                the output extent E, F must be >= 1
 *   rowptr[M+1]  rowptr[0] == 0, non-decreasing; nnz = rowptr[M] < 2^31
 *   colidx[nnz]  column in [0, C*R*S); any order within a row; no duplicates
 *   value[nnz]   fp32 weights (explicit zeros are allowed)
 *   stream       stream for the upload; the call waits for it before returning
 * Output: *out receives a new handle (device buffers on the current device).
 * Errors: INVALID_ARG, BAD_CSR, UNSUPPORTED, ALLOC, CUDA; *out is untouched.
 */
int spconv_pack(int C, int H, int W, int M, int R, int S, int stride, int pad,
                const int32_t *rowptr, const int32_t *colidx, const float *value,
                void *stream, spconv_packed **out);

/* Packed weight formats of spconv_pack_ex. */
typedef enum spconv_format {
    SPCONV_FORMAT_F32 = 0,      /* 8-byte entries: fp32 value + int32 precomputed offset    */
    SPCONV_FORMAT_PACKED32 = 1, /* 4-byte words of the first page's Sec. 5.3 / Fig. 4:      */
                                /* [31:16] FP16 value, [15:8] input channel (within the     */
                                /* chunk), [7:4] kernel column, [3:0] kernel row; R, S <= 16 */
    SPCONV_FORMAT_WS = 2,       /* weight-stationary mapping of Escoin (arXiv 1802.10280),  */
                                /* Figs. 5-7: one output channel per thread block, its      */
                                /* entries staged in shared memory, the input read in place */
                                /* through the read-only cache.  8-byte entries {fp32 value, */
                                /* uint32 word = off << 8 | r << 4 | s} with the stretched   */
                                /* offset off = c*H*W + r*W + s; R, S <= 16 and             */
                                /* C*H*W + R*W + S <= 2^24; forwards take N <= 65535         */
} spconv_format;

/*
 * spconv_pack_ex -- spconv_pack with a choice of entry format, a batch-size
 * hint for the tiling plan, and of where the handle lives.
 *   format      spconv_format (PACKED32 rounds every weight to FP16 once,
 *               round-to-nearest-even, and halves the sparse entry stream;
 *               dense rows keep their FP16-rounded values as fp32)
 *   batch_hint  batch size the forwards will mostly use (0 = unknown).  It
 *               only shapes the plan (output channels per warp, channel chunk
 *               size); forwards accept any N either way.
 *   host_only   != 0: as spconv_pack_host (no device work, stream ignored)
 * Errors as spconv_pack; INVALID_ARG for an unknown format or a negative
 * batch_hint, UNSUPPORTED for PACKED32 or WS with R or S > 16, for WS with
 * C*H*W + R*W + S > 2^24.  spconv_forward(_ex) on a WS handle runs
 * the weight-stationary kernel and returns UNSUPPORTED for N > 65535.
 */
int spconv_pack_ex(int C, int H, int W, int M, int R, int S, int stride, int pad,
                   const int32_t *rowptr, const int32_t *colidx, const float *value, int format,
                   int batch_hint, int host_only, void *stream, spconv_packed **out);

/*
 * spconv_forward -- Y = conv(X, packed weights); the hot path.
 *
 * Launches the sparse direct convolution kernel on `stream` and returns
 * without synchronising.  Y is overwritten (no accumulation, no bias).
 * An output channel whose CSR row is empty is written as zeros.
 *   N                 batch size (>= 0; N == 0 is a no-op)
 *   C,H,W,M,R,S,stride,pad   must equal the values given to spconv_pack
 *   input   device pointer, N*C*H*W floats, 16-byte aligned
 *   packed  handle from spconv_pack (read-only; may be shared by concurrent
 *           forwards on different streams)
 *   output  device pointer, N*M*E*F floats, 4-byte aligned, not overlapping input
 * Errors: INVALID_ARG (NULL/misaligned/negative N), MISMATCH (shape or current
 * device differs from the handle's), UNSUPPORTED, CUDA (launch failure).
 * Inputs are expected to be finite.
 */
int spconv_forward(int N, int C, int H, int W, int M, int R, int S, int stride, int pad,
                   const float *input, const spconv_packed *packed, float *output,
                   void *stream);

/* Activations of the fused epilogue of spconv_forward_ex. */
typedef enum spconv_act { SPCONV_ACT_NONE = 0, SPCONV_ACT_RELU = 1 } spconv_act;

/*
 * spconv_forward_ex -- spconv_forward with a fused epilogue applied in the
 * kernel's write-back:  Y[n,m,e,f] = act(conv[n,m,e,f] + bias[m]).
 * (The first page names bias/activation fusion and layer chaining as its
 * follow-on work, Sec. 7.)
 *   bias  device pointer to M floats (4-byte aligned), or NULL for no bias
 *   act   SPCONV_ACT_NONE or SPCONV_ACT_RELU (y = max(y, 0))
 * Every other argument, and the errors, as for spconv_forward; INVALID_ARG
 * also for an unknown act or a bias overlapping the output.
 */
int spconv_forward_ex(int N, int C, int H, int W, int M, int R, int S, int stride, int pad,
                      const float *input, const spconv_packed *packed, const float *bias,
                      int act, float *output, void *stream);

/*
 * spconv_forward_host -- spconv_forward_ex with the activation and the result
 * in host memory, enqueued on `stream` by one call; nothing is allocated.
 * When CUDA maps both host buffers for the current device (page-locked memory
 * from cudaHostAlloc / cudaHostRegister, each inside one allocation): a copy
 * kernel reads input_host through its device mapping into dev_input; the
 * forward (launched behind it with programmatic dependent launch) writes a Y
 * of at most 1 MiB straight into output_host through its mapping (dev_output
 * is not touched), a larger Y into dev_output, which a second copy kernel
 * writes to output_host.  Otherwise: cudaMemcpyAsync of input_host into
 * dev_input, the forward into dev_output, cudaMemcpyAsync of dev_output into
 * output_host.
 *   input_host   host pointer, N*C*H*W floats (NCHW); page-locked for the
 *                work to be asynchronous (pageable memory takes the copy path,
 *                where CUDA may copy before the call returns)
 *   output_host  host pointer, N*M*E*F floats, 4-byte aligned, page-locked
 *                likewise; must not overlap input_host
 *   dev_input    device workspace, N*C*H*W floats, 16-byte aligned
 *   dev_output   device workspace, N*M*E*F floats, 4-byte aligned, not
 *                overlapping dev_input; its contents afterwards are unspecified
 *   bias, act    as for spconv_forward_ex (bias is a device pointer or NULL)
 * Asynchronous: output_host holds Y once the stream has passed the call's
 * work; the caller keeps all four buffers alive until then.  Errors: those of
 * spconv_forward_ex (with dev_input / dev_output in the roles of input /
 * output), INVALID_ARG for a NULL, misaligned or overlapping host buffer, all
 * returned before anything is enqueued; CUDA when a copy or a launch cannot be
 * enqueued (work already enqueued is not undone).  N = 0 is a no-op.
 */
int spconv_forward_host(int N, int C, int H, int W, int M, int R, int S, int stride, int pad,
                        const float *input_host, const spconv_packed *packed, const float *bias,
                        int act, float *output_host, float *dev_input, float *dev_output,
                        void *stream);

/* Bytes of device memory behind spconv_forward_host_noalloc's workspaces. */
#define SPCONV_NOALLOC_MAX_BYTES (32u << 20)

/*
 * spconv_forward_host_noalloc -- spconv_forward_host without the two device
 * workspace arguments, for callers that must not allocate device memory at
 * the time they run a layer: a plugin inside a framework whose allocator owns
 * the GPU's memory, a service whose memory is budgeted up front, or a caller
 * on a latency-critical path that cannot take cudaMalloc's implicit
 * synchronisation.  (No counterpart in the papers: this is an interface
 * convenience.)  The call allocates nothing -- no cudaMalloc, cudaFree or
 * allocating library routine; the packed weights come from an earlier
 * spconv_pack, which does allocate, once, at set-up.
 *
 * The workspaces are one statically declared device array of
 * SPCONV_NOALLOC_MAX_BYTES (32 MiB), which every GPU that loads this code
 * holds until the process exits: the staged input (N*C*H*W floats) at its
 * start and, 256-byte aligned after it, the staged output (N*M*E*F floats;
 * used only when Y exceeds 1 MiB or the host buffers are not mapped).
 *   Arguments, work enqueued, asynchrony and errors: as spconv_forward_host.
 *   Also UNSUPPORTED when the two workspaces do not fit in the array
 *   (rounding the input to 256 bytes), INVALID_ARG for a non-positive shape
 *   argument, and CUDA when the array's address cannot be looked up.
 *   Set-up: the first call on each device (with that device current) looks up
 *   the array's device address with cudaGetSymbolAddress; make that first call
 *   before any stream capture.
 *   Sharing: every call on a device uses the same array, and it keeps the last
 *   call's contents (each call overwrites all it reads).  Calls whose work
 *   overlaps on the GPU -- on different streams, or from different threads --
 *   race on the array: order them on one stream or by events.
 */
int spconv_forward_host_noalloc(int N, int C, int H, int W, int M, int R, int S, int stride,
                                int pad, const float *input_host, const spconv_packed *packed,
                                const float *bias, int act, float *output_host, void *stream);

/* Frees the handle and its device buffers.  NULL-safe.  The caller must make
 * sure no forward that uses the handle is still running. */
void spconv_packed_free(spconv_packed *p);

/* Static, never-NULL description of a status code. */
const char *spconv_status_string(int status);

/*
 * spconv_pack_host -- the same packing as spconv_pack, kept in host memory
 * only (no device work, no GPU needed).  The handle can be inspected with
 * spconv_packed_info / spconv_packed_copy_array; spconv_forward rejects it
 * with SPCONV_ERR_MISMATCH.  Same arguments and errors as spconv_pack.
 */
int spconv_pack_host(int C, int H, int W, int M, int R, int S, int stride, int pad,
                     const int32_t *rowptr, const int32_t *colidx, const float *value,
                     spconv_packed **out);

/*
 * spconv_device_status -- failures that kernels using this handle recorded on
 * the device.  Synchronises `stream`, reads and clears the handle's device
 * error word and returns SPCONV_OK if it was clear, SPCONV_ERR_DEVICE if not
 * (then *flags, if not NULL, receives the bits: 1 = a pipeline wait in the
 * forward kernel ran out its time limit and the kernel returned without
 * writing its outputs; 2 = after such a timeout, the wait for the block's
 * copies still in flight ran out as well, so an asynchronous copy may have
 * landed in shared memory after the block left: treat the CUDA context as
 * suspect and reset it before further use; 4 = only in the bounds-checked
 * build libspconv_debug.so: an access failed its bounds check and was
 * skipped, so the outputs are not valid).  Errors: INVALID_ARG (NULL or
 * host-only handle), CUDA.
 */
int spconv_device_status(const spconv_packed *p, void *stream, int32_t *flags);

/*
 * spconv_selftest_wait -- exercises, on the current device, the bounded wait
 * the forward kernel uses for its copy pipeline: a one-warp kernel waits on a
 * shared-memory barrier with a 20 ms limit.  complete = 0 leaves the barrier
 * incomplete, so the wait runs out, the kernel records the timeout and
 * returns (the context stays usable); complete != 0 completes it first.
 * Synchronises `stream`.  *flags receives bit 0 (timed out) / bit 1
 * (completed).  Returns SPCONV_ERR_DEVICE when the wait timed out, SPCONV_OK
 * when it completed; INVALID_ARG (flags NULL), ALLOC, CUDA.
 */
int spconv_selftest_wait(int complete, void *stream, int32_t *flags);

/*
 * spconv_trace_read -- the per-block timeline of the last spconv_forward /
 * spconv_forward_ex launch on the current device, recorded only by the trace
 * build libspconv_trace.so (the same sources compiled with -DSPCONV_TRACE=1);
 * no counterpart in the pages, a diagnostic of this library.  Copies up to
 * `bytes` to host_dst: 4 x uint64 per block in launch order (linear block
 * index y * grid_x + x, the first 65536 blocks): start, first stage ready,
 * end of the chunk pipeline (global-timer ns; 0 = not reached), and
 * smid | group << 16 | group flags << 32.  Synchronises the device.  Errors:
 * INVALID_ARG (NULL or negative size), UNSUPPORTED (not the trace build),
 * CUDA.
 */
int spconv_trace_read(void *host_dst, int64_t bytes);

/* Geometry and sizes of a packed handle (all counts are plain integers). */
typedef struct spconv_packed_info {
    int32_t C, H, W, M, R, S, stride, pad, E, F;
    int64_t nnz;            /* nonzeros of the CSR input                        */
    int64_t entries;        /* packed (value, offset) entries (== nnz)          */
    int32_t tile_rows;      /* output rows each lane carries                    */
    int32_t shift;          /* staged column of a tile's first input column     */
    int32_t tile_cols;      /* output columns per tile (lanes per lane row)     */
    int32_t tiles_y, tiles_x;
    int32_t in_rows;        /* staged input rows per channel (with halo)        */
    int32_t in_cols;        /* staged input columns per channel (with halo)     */
    int32_t phase_pitch;    /* words per stride-phase sub-row                   */
    int32_t row_pitch;      /* words per staged input row                       */
    int32_t plane;          /* words per staged channel                         */
    int32_t chunk;          /* input channels staged at once                    */
    int32_t num_chunks;
    int32_t slots_per_warp; /* output channels a warp carries at once           */
    int32_t warps;          /* warps per block                                  */
    int32_t groups;         /* output-channel groups (blocks along grid y)      */
    int32_t num_slots;      /* groups * warps * slots_per_warp                  */
    int32_t on_device;      /* 1 if device buffers exist (spconv_pack)          */
    int64_t device_bytes;   /* bytes of device memory held by the handle        */
    int64_t smem_bytes;     /* dynamic shared memory per block of the forward   */
    int64_t max_warp_nnz;   /* heaviest warp's total entries (balance metric)   */
    int64_t mean_warp_nnz;  /* mean over non-empty warps, rounded down          */
    int32_t hdr_words;      /* 32-bit words of a weight blob's header           */
    int32_t blob_stage_bytes; /* largest weight blob (bytes, rounded to 128)    */
    int32_t in_stage_bytes;   /* staged input of one chunk (bytes, to 128)      */
    int32_t lane_rows;        /* lane rows of a warp (output rows per tile =    */
                              /* lane_rows * tile_rows)                         */
    int32_t dense_groups;     /* leading groups whose blobs are dense-tap       */
    int32_t dense_mask_words; /* words of a dense blob's slot masks            */
    int32_t format;           /* spconv_format of the sparse entries           */
    int32_t batch_hint;       /* batch size the plan targets (0 = unknown)     */
    int32_t blob_stride;      /* bytes between consecutive blobs when they are  */
                              /* stored at a fixed stride (nearly equal sizes,  */
                              /* each padded to the largest), else 0            */
    int32_t tap_pairs;        /* 1: sparse blobs also hold pair entries (see   */
                              /* SPCONV_ARRAY_BLOBS)                           */
    int32_t plane_stage;      /* 1: the forward stages raw input planes (pitch */
                              /* W after 16 zeroed words); F32 entry offsets   */
                              /* are then (16 + c*H*W + (r-1)*W + (s-1)) << 4  */
                              /* | flags: bit 0 s == 0, 1 s == 2, 2 r == 0,    */
                              /* 3 r == 2                                      */
    int32_t col_blocks;       /* 1: column blocks -- a tile is lane_rows rows  */
                              /* of tile_cols outputs, each lane holding       */
                              /* tile_rows consecutive outputs of one row      */
                              /* (entry offsets as for the padded tile)        */
    int32_t tile_images;      /* 2: image-pair column blocks -- lanes 0..3 of  */
                              /* a lane row on image 2n, lanes 4..7 on image   */
                              /* 2n + 1; a stage holds both images' sub-tiles  */
                              /* (same offsets), the second pair_off words     */
                              /* after the first; else 1                       */
    int32_t pair_off;
} spconv_packed_info;

/* For a SPCONV_FORMAT_WS handle: tile_rows, lane_rows, tile_cols, tiles_y and
 * tiles_x describe one block's output tile (warps * lane_rows * tile_rows rows
 * of tile_cols columns); chunk = entries per pipeline stage, num_chunks = the
 * most stages of any row; max_warp_nnz / mean_warp_nnz = the longest / mean
 * row (one row per block); the input-staging fields are 0. */
int spconv_packed_info_get(const spconv_packed *p, spconv_packed_info *info);

/* How spconv_forward would launch for a batch of N images (host logic only;
 * no device work).  TMA staging also needs the input pointer's tensor map to
 * encode, which this query does not try. */
typedef struct spconv_launch_info {
    int32_t kernel;          /* 0: tiled kernel, 1: weight-stationary kernel     */
    int32_t grid_x, grid_y, grid_z;
    int32_t block_threads;
    int32_t cluster;         /* blocks per cluster splitting the channel chunks  */
    int32_t push;            /* 1: the cluster reduces by remote stores into the */
                             /* owning block (one cluster barrier), 0: by remote */
                             /* reads (two barriers) or no cluster              */
    int32_t group_fast;      /* 1: all channel groups of a tile run together     */
    int32_t tma;             /* 1: input staged by TMA tensor copies             */
    int32_t pdl;             /* 1: launched with programmatic stream             */
                             /* serialization (start-up overlaps the previous    */
                             /* kernel on the stream; input and output are only  */
                             /* touched after that kernel has completed)         */
    int64_t smem_bytes;      /* dynamic shared memory per block                  */
} spconv_launch_info;

/* Fills *info for a forward of N >= 1 images with handle p.  INVALID_ARG (NULL,
 * N < 1), UNSUPPORTED (a grid spconv_forward would reject). */
int spconv_launch_info_get(const spconv_packed *p, int N, spconv_launch_info *info);

/* Which host-side array spconv_packed_copy_array copies. */
typedef enum spconv_array {
    SPCONV_ARRAY_BLOBS = 0,    /* the weight blobs, one per (group, chunk), each    */
                               /* 16-byte aligned.  Sparse groups: hdr_words       */
                               /* uint32 entry indices (slot w*Q+q spans           */
                               /* [hdr[w*Q+q], hdr[w*Q+q+1])), then entries of     */
                               /* {float value, int32 offset} (F32) or 32-bit      */
                               /* packed words (PACKED32).  With tap_pairs (F32,   */
                               /* Q = 2 or 4 slots per warp, NP = Q(Q-1)/2): next  */
                               /* come warps*NP + 1 words hp of pair ranges in     */
                               /* 8-byte units -- warp w's pair p (slots q1 < q2,  */
                               /* numbered in lexicographic order) spans           */
                               /* [hp[w*NP+p], hp[w*NP+p+1]) -- and the pair       */
                               /* entries are 16 bytes {float value of q1, float   */
                               /* value of q2, int32 offset, 0}: a tap both slots  */
                               /* use, from a 16-byte boundary.  Dense groups:     */
                               /* dense_mask_words uint32 slot masks [warp][chan], */
                               /* then floats [warp][chan][slot][R*S rounded to 4] */
    SPCONV_ARRAY_BLOB_OFF = 1, /* uint32 [groups * num_chunks + 1]: blob starts in  */
                               /* 16-byte units                                     */
    SPCONV_ARRAY_SLOT_OC = 2,  /* int32 [num_slots]: output channel of a head slot,  */
                               /* -1 for empty slots and later parts of split rows */
                               /* SPCONV_FORMAT_WS instead: BLOBS = the entries of  */
                               /* every row in column order, each row starting on an */
                               /* even entry; BLOB_OFF = uint32 [2 * M] (first entry, */
                               /* entry count) of row m; SLOT_OC = int32 [M] the row */
                               /* of each block column (heaviest first); SLOT_NEXT   */
                               /* and GROUP_FLAGS are empty                          */
    SPCONV_ARRAY_SLOT_NEXT = 3,/* int32 [num_slots]: group-local slot of the next   */
                               /* part of the same output channel, or -1            */
    SPCONV_ARRAY_GROUP_FLAGS = 4 /* int32 [groups]: bit 0 dense-tap blobs, bit 1    */
                               /* the group has split rows                          */
} spconv_array;

/* Copies one packed array into dst (host, dst_bytes long).  *needed (if not
 * NULL) receives the array's size in bytes.  INVALID_ARG if dst_bytes is too
 * small (dst may be NULL to query the size). */
int spconv_packed_copy_array(const spconv_packed *p, int which, void *dst, int64_t dst_bytes,
                             int64_t *needed);

#ifdef __cplusplus
}
#endif

#endif /* SPCONV_H */
