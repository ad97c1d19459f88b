/*
 * ulysses.h -- C ABI of the GB300 Ulysses 4D sequence/head relayout library (libulysses.so).
 *
 * What the library computes (fast-ulysses 0.1.0, PyPI page, opening paragraph and "Quick start";
 * fast-ulysses 0.2.1, README, "Quick start" and "API"): the all-to-all of Ulysses sequence
 * parallelism on W ranks, here W virtual ranks on one GPU, each rank a separate device buffer.
 * With s_q = seq_splits[q], n_r = head_splits[r], S = sum s_q, N = sum n_r,
 * seq_off(q) = s_0 + ... + s_(q-1) and head_off(r) = n_0 + ... + n_(r-1):
 *
 *   mode 0  rank q's (b, s_q, N, d) tensor  ->  rank r's (b, S, n_r, d) tensor
 *           out[r][bb][seq_off(q) + i][h][:] = in[q][bb][i][head_off(r) + h][:]
 *   mode 1  the exact inverse on the same splits ("a second trades it back"):
 *           out[q][bb][i][head_off(r) + h][:] = in[r][bb][seq_off(q) + i][h][:]
 *
 * Uneven shards (fast-ulysses 0.1.0, "What it does") are the general case; even splits are not a
 * separate path. A split of zero is allowed (that rank contributes or receives nothing); S and N
 * must be positive.
 *
 * Conventions shared by every entry point:
 *  - Every function returns a status: ULY_OK (0) or a negative ULY_E* code; ulysses_strerror()
 *    names it. Nothing is printed and nothing aborts.
 *  - Tensors are dense, row-major (C order), as the shapes above state, with no padding.
 *  - Device pointers are addresses on the current CUDA device, 16-byte aligned (ULY_EALIGN
 *    otherwise). A pointer may be NULL only when that rank's tensor has zero bytes.
 *  - The caller owns every buffer and keeps it alive until the work queued on `stream` has
 *    finished. Pointer arrays (W entries each) are read during the call only.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Device work is
 *    queued asynchronously; no call synchronises except ulysses_device_status().
 *  - Calls allocate no memory. A plan holds only host memory and may be used by several host
 *    threads at once for launches; ulysses_plan_set_chunk_bytes() must not race with launches.
 *  - Input and output ranges must not overlap each other, and outputs must not overlap one another
 *    (ULY_EOVERLAP).
 *  - Kernels never spin without bound: a wait that exceeds its time limit sets a bit in a device
 *    status word, read with ulysses_device_status().
 */
#ifndef ULYSSES_H
#define ULYSSES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
    ULY_OK = 0,
    ULY_EINVAL = -1,   /* bad argument: W, splits, b, d, dtype, mode, rank, NULL pointer */
    ULY_EALIGN = -2,   /* a device pointer is not 16-byte aligned, or d * elem_size % 16 != 0 */
    ULY_EOVERLAP = -3, /* an output range overlaps an input range or another output range */
    ULY_ECHUNK = -4,   /* the chunk cap is smaller than one sequence row on some rank */
    ULY_ECUDA = -5,    /* a CUDA runtime call failed; ulysses_last_cuda_error() has the code */
    ULY_ENOMEM = -6,   /* host memory for a plan could not be allocated */
    ULY_EDEVICE = -7,  /* a kernel recorded a wait timeout in the device status word */
    ULY_ESCRATCH = -8  /* the call needs more scratch than the library's static array holds */
};

/* Element types (fast-ulysses 0.2.1, README, "Limits": float16 / bfloat16 / float32 /
 * float8_e4m3fn / float8_e5m2 / int8 / uint8). The relayout moves bytes, so only the size
 * matters to it; the fused QK calls require ULY_BF16 or ULY_F16. */
enum {
    ULY_U8 = 1,
    ULY_F8E4M3 = 2,
    ULY_F8E5M2 = 3,
    ULY_I8 = 4,
    ULY_F16 = 5,
    ULY_BF16 = 6,
    ULY_F32 = 7
};

/* RoPE pair layouts of the fused QK calls (ulysses_plan_set_rope_pairs): pair j is
 * (x[2j], x[2j+1]) (ULY_ROPE_ADJACENT, the default) or (x[j], x[j + d/2]) (ULY_ROPE_HALF, the
 * "rotate half" layout); both rotate pair j by p * rope_theta^(-2j/d). The pages name the fused
 * QK RMSNorm + RoPE without fixing its layout; both common ones are provided. */
enum { ULY_ROPE_ADJACENT = 0, ULY_ROPE_HALF = 1 };

/* Relayout engines: ULY_ENGINE_AUTO picks the faster measured kernel for the plan: the tensor
 * engine when every head group's run (n_r * d * elem_size) has the same length of at most 2048
 * bytes, or when the plan's CTA cap (ulysses_plan_set_max_ctas) is below the SM count and every
 * run is at most 2048 bytes; the TMA kernel otherwise.
 * ULY_ENGINE_CE issues one pitched cudaMemcpy2DAsync per (source shard, destination rank, batch
 * index) on the copy engines, no kernel: the pages' own transport design (fast-ulysses 0.1.0,
 * opening paragraph: pitched 2D/3D copies on the copy engines) run between buffers of one GPU,
 * kept for comparison and for overlapping with SM-bound work. ULY_ENGINE_TENSOR moves each
 * (source shard, destination rank) block of up to 256 rows with one tiled tensor-map copy on its
 * strided side and one bulk copy on its contiguous side (fewer copy instructions per byte than
 * the TMA kernel's one per row; one CTA per SM); plans with a run above 2048 bytes use the TMA
 * kernel instead. Every engine gives the same bytes. */
enum { ULY_ENGINE_AUTO = 0, ULY_ENGINE_TMA = 1, ULY_ENGINE_VEC = 2, ULY_ENGINE_CE = 3,
       ULY_ENGINE_TENSOR = 4 };

typedef struct ulysses_plan_s* ulysses_plan_t;

/*
 * Build the host-side addressing plan (fast-ulysses 0.1.0, "What it does": the addressing is a
 * host-side plan, testable without a GPU, with no launch configuration to tune).
 *   W            number of ranks, 1..8 (fast-ulysses 0.1.0, "Limits": world_size in [1, 8],
 *                odd sizes included).
 *   b            batch, >= 1.
 *   seq_splits   W entries s_q >= 0 with S = sum > 0 (host array, read during the call).
 *   head_splits  W entries n_r >= 0 with N = sum > 0 (host array, read during the call).
 *   d            head dimension; d * elem_size must be a multiple of 16 (fast-ulysses 0.2.1,
 *                "Limits": d * elem_size 16-byte aligned), else ULY_EALIGN.
 *   dtype        one of ULY_U8 .. ULY_F32.
 *   out          receives the plan; release it with ulysses_plan_destroy().
 * Makes no CUDA call. The default chunk cap is 1 GiB (see ulysses_plan_set_chunk_bytes).
 */
int ulysses_plan(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits, int64_t d,
                 int dtype, ulysses_plan_t* out);

/* Release a plan (NULL is accepted). Work already queued with it is unaffected. */
int ulysses_plan_destroy(ulysses_plan_t plan);

/*
 * Cap on the bytes any one rank reads or writes in one kernel launch (FastVideo, "Ulysses
 * performance on GB200": each rank keeps at most 1 GiB of window storage and long sequences are
 * exchanged in chunks). A call whose per-rank bytes exceed the cap is split into several launches
 * along the sequence shards (the source sequence in mode 0, the destination sequence in mode 1);
 * the result is identical to one launch. max_chunk_bytes >= 1; default 1 << 30.
 */
int ulysses_plan_set_chunk_bytes(ulysses_plan_t plan, int64_t max_chunk_bytes);

/*
 * Cap on the CTAs (thread blocks) of every kernel launched with this plan; 0 (the default)
 * means no cap: the kernels' persistent grids cover every SM. A cap leaves the remaining SMs
 * free for work on other streams (a GEMM, attention) at the cost of this call's bandwidth; it
 * changes no result. The pages have no such setting (their transfer runs on copy engines, which
 * use no SMs); it exists for overlapping the relayout with compute on one GPU.
 * max_ctas >= 0. Like the chunk cap, it must not race with launches using the plan.
 */
int ulysses_plan_set_max_ctas(ulysses_plan_t plan, int64_t max_ctas);

/* Kernel of the fused forward calls (ulysses_a2a_4d_qk_fused, its host-buffer form, and the
 * packed forms ulysses_a2a_4d_qkv_fused / ulysses_a2a_4d_packed_fused) made with this plan, and
 * of their backward (see ulysses_plan_fused_backward_kernel for its automatic choice): ULY_ENGINE_TMA, units of whole tokens (one bulk
 * copy in per tensor, one out per (token, tensor, destination rank)); ULY_ENGINE_TENSOR, units of
 * a block of whole rows (one tiled tensor-map copy in per tensor that lands the rows grouped by
 * destination rank, one bulk copy out per (tensor, rank)), for plans whose head groups all have
 * the same run n * d * elem_size of at most 2048 bytes (other plans use the token units);
 * ULY_ENGINE_AUTO (the default) takes the tensor-map kernel where it fits, d is a power of two
 * and a row (N * d * elem_size) is at most 10,240 bytes, where it measured faster, else the
 * token units.
 * All give the same bytes. The setting applies to the packed calls too (their q and k planes as
 * above, the other planes moved in blocks of 2R rows). ULY_EINVAL for another engine. Must not
 * race with launches using the plan. */
int ulysses_plan_set_fused_engine(ulysses_plan_t plan, int engine);

/* The kernel that a fused forward call (separate or packed inputs) takes for this plan, after
 * its fused-engine setting: ULY_ENGINE_TENSOR (row blocks through tensor maps) or ULY_ENGINE_TMA
 * (token units). No CUDA call. ULY_EINVAL for a null plan or engine pointer. */
int ulysses_plan_fused_kernel(ulysses_plan_t plan, int* engine);

/* The same for the backward of the fused call (ulysses_a2a_4d_qk_fused_backward and its packed
 * and static forms): ULY_ENGINE_TENSOR, units of whole-row blocks whose forward input arrives
 * through one tiled tensor-map copy grouped by head group and whose gradient rows arrive as one
 * span per rank; or ULY_ENGINE_TMA, token units. The plan's fused-engine setting applies; under
 * ULY_ENGINE_AUTO the backward takes row blocks where they fit (equal head groups, runs of at
 * most 2048 bytes) and a row N * d * elem_size is at least 6,144 bytes, where they measured
 * faster. No CUDA call. ULY_EINVAL for a null plan or engine pointer. */
int ulysses_plan_fused_backward_kernel(ulysses_plan_t plan, int* engine);

/* RoPE pair layout (ULY_ROPE_ADJACENT or ULY_ROPE_HALF) of the fused calls made with this plan:
 * the forward, the interleaved QKV form, the host-buffer form and the backward. Default
 * ULY_ROPE_ADJACENT. Must not race with launches using the plan. */
int ulysses_plan_set_rope_pairs(ulysses_plan_t plan, int pairs);

/* Bytes of rank `rank`'s input and output tensors for `mode` (either pointer may be NULL). */
int ulysses_plan_bytes(ulysses_plan_t plan, int mode, int rank, int64_t* in_bytes,
                       int64_t* out_bytes);

/* The engine that a call with ULY_ENGINE_AUTO takes for this plan on the calling thread's
 * current device: ULY_ENGINE_TENSOR or ULY_ENGINE_TMA (see the engine list above), from the
 * plan's splits, element size and CTA cap and the device's SM count. ULY_EINVAL for a null plan
 * or engine pointer; a CUDA error status when the device cannot be queried. */
int ulysses_plan_auto_engine(ulysses_plan_t plan, int* engine);

/* Number of launches a call in `mode` makes under the current chunk cap (ULY_ECHUNK when no
 * split along whole sequence rows meets the cap). */
int ulysses_plan_num_chunks(ulysses_plan_t plan, int mode, int64_t* n_chunks);

/* Rows of each sequence shard that launch `chunk` covers: for q < W, rows
 * [row_lo[q], row_lo[q] + row_count[q]) of shard q (host arrays of W entries). */
int ulysses_plan_chunk_rows(ulysses_plan_t plan, int mode, int64_t chunk, int64_t* row_lo,
                            int64_t* row_count);

/*
 * One rank's share of the exchange, for a transport that runs the ranks on separate GPUs
 * (fast-ulysses 0.1.0, opening paragraph: pitched peer copies into the other ranks' windows).
 * This library runs all W ranks on one GPU and issues no such copies; the description lets a
 * multi-GPU caller (or a test) move each rank's bytes itself with the same plan.
 * A segment is a strided block: for every batch index bb < b and row i < rows, the row_bytes at
 *   src_offset + bb * src_batch_pitch + i * src_row_pitch   of the sending rank's tensor go to
 *   dst_offset + bb * dst_batch_pitch + i * dst_row_pitch   of rank `peer`'s tensor.
 * Tensors are those of ulysses_a2a_4d in `mode`: in mode 0 a rank sends from its (b, s_q, N, d)
 * input to every rank's (b, S, n_r, d) output; in mode 1 from its (b, S, n_r, d) input to every
 * rank's (b, s_q, N, d) output.
 */
typedef struct {
    int64_t peer;             /* the receiving rank */
    int64_t rows;             /* rows per batch index (0: nothing to send) */
    int64_t row_bytes;        /* bytes of one row */
    int64_t src_offset;       /* byte offset of row 0, batch index 0, in the sender's tensor */
    int64_t src_row_pitch;    /* bytes between consecutive rows there */
    int64_t src_batch_pitch;  /* bytes between consecutive batch indices there */
    int64_t dst_offset;       /* the same three in the receiver's tensor */
    int64_t dst_row_pitch;
    int64_t dst_batch_pitch;
} ulysses_segment_t;

/* Fill segs[0 .. W-1] with the segments rank `rank` sends in `mode` (segs[r] goes to rank r,
 * itself included). Host only: makes no CUDA call. Together the W ranks' segments move every
 * byte of the relayout once. */
int ulysses_plan_rank_segments(ulysses_plan_t plan, int mode, int rank, ulysses_segment_t* segs);

/*
 * The relayout (fast-ulysses 0.2.1, README, "API": all_to_all_4d(x, mode, seq_splits,
 * head_splits)), for all W ranks in one call.
 *   mode     0 or 1 (see the top of this file).
 *   in_ptrs  W device pointers; mode 0: rank q's (b, s_q, N, d), mode 1: rank r's (b, S, n_r, d).
 *   out_ptrs W device pointers; mode 0: rank r's (b, S, n_r, d), mode 1: rank q's (b, s_q, N, d).
 * Bit-exact byte move. Queues one kernel launch per chunk on `stream`.
 */
int ulysses_a2a_4d(ulysses_plan_t plan, int mode, const void* const* in_ptrs,
                   void* const* out_ptrs, void* stream);

/* Same as ulysses_a2a_4d with an explicit engine (ULY_ENGINE_*): TMA bulk copies through shared
 * memory, 16-byte vector loads and stores, or copy-engine pitched copies. All give identical
 * bytes. With ULY_ENGINE_CE the call queues W * W * b copies per chunk (fewer when a split is
 * zero) and no kernel. */
int ulysses_a2a_4d_engine(ulysses_plan_t plan, int mode, int engine, const void* const* in_ptrs,
                          void* const* out_ptrs, void* stream);

/*
 * Mode 0 with QK RMSNorm + RoPE applied inside the scatter (fast-ulysses 0.1.0, "Fusion
 * examples"). For q and k separately, every head row x of d values at global sequence
 * position p = seq_off(q) + i becomes
 *     y = x / sqrt(mean(x^2) + eps) * w                  (w: rms_w[0][:] for q, rms_w[1][:] for k)
 *     pair j of y rotated by the angle p * rope_theta^(-2j/d), j < d/2 (pairs (y[2j], y[2j+1]),
 *     or (y[j], y[j + d/2]) after ulysses_plan_set_rope_pairs(plan, ULY_ROPE_HALF))
 * computed in fp32 and rounded once to the element type (nearest even), then placed where mode 0
 * puts it.
 *   plan     must have dtype ULY_BF16 or ULY_F16, d a multiple of 8 from 8 to 256 (e.g. 64,
 *            72, 80, 96, 128), S < 2^24.
 *   q_in, k_in     W device pointers, rank q's (b, s_q, N, d) elements of the plan's dtype.
 *   q_out, k_out   W device pointers, rank r's (b, S, n_r, d), same dtype.
 *   rms_w    device pointer to 2 * d fp32 values, q's weight then k's.
 *   eps      > 0 or 0; rope_theta > 0.
 * V and the attention output go through ulysses_a2a_4d (mode 0 / mode 1).
 */
int ulysses_a2a_4d_qk_fused(ulysses_plan_t plan, const void* const* q_in, const void* const* k_in,
                            void* const* q_out, void* const* k_out, const float* rms_w, float eps,
                            float rope_theta, void* stream);

/*
 * Backward of ulysses_a2a_4d_qk_fused on the same plan. The relayout is differentiable and its
 * backward uses the plan saved by the forward (fast-ulysses 0.2.1, README, "Quick start" and
 * "Limits"; FastVideo, "Ulysses performance on GB200"); the backward of mode 0 is mode 1 (the
 * plain relayout's gradient is ulysses_a2a_4d with mode 1). Here the vector-Jacobian product of
 * the RMSNorm + RoPE transform is applied inside that mode-1 gather. For q and k separately, per
 * head row x at global position p with output gradient gy (the row mode 0 made of x):
 *     r = 1 / sqrt(mean(x^2) + eps),  u = gy rotated back by p * rope_theta^(-2j/d) per pair j,
 *     dx = r * (u * w - x * r * <u * w, x * r> / d)      -> dq_out / dk_out, rounded once
 *     dw = sum over all rows of all ranks of u * x * r   -> dw[0][:] (q), dw[1][:] (k), fp32
 * computed in fp32 (the sums over rows in fp32, in an order that does not depend on timing).
 *   dq_out, dk_out  W device pointers, rank q's (b, s_q, N, d) of the plan's dtype (bf16 or
 *                   fp16; the forward's inputs' shape). The pair layout is the plan's.
 *   q_in, k_in      W device pointers, the forward's inputs (rank q's (b, s_q, N, d)).
 *   dq_in, dk_in    W device pointers, gradients of the forward's outputs, rank r's (b, S, n_r, d).
 *   rms_w           device pointer, 2 * d fp32 (as the forward); dw: device pointer, 2 * d fp32,
 *                   overwritten.
 *   eps, rope_theta, plan requirements: as ulysses_a2a_4d_qk_fused.
 *   workspace       device memory of at least ulysses_qk_fused_backward_workspace bytes, 16-byte
 *                   aligned, the caller's; partial sums of dw live there while the call runs, so
 *                   two calls in flight at once need two workspaces. No initial contents needed.
 * Queues two launches per chunk on `stream`. ULY_EINVAL for a short workspace; outputs (with dw
 * and the workspace) may not overlap inputs or each other (ULY_EOVERLAP).
 */
int ulysses_a2a_4d_qk_fused_backward(ulysses_plan_t plan, void* const* dq_out, void* const* dk_out,
                                     const void* const* q_in, const void* const* k_in,
                                     const void* const* dq_in, const void* const* dk_in,
                                     const float* rms_w, float* dw, float eps, float rope_theta,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes ulysses_a2a_4d_qk_fused_backward needs for `plan` on the current device (one
 * 2 * d fp32 slot per CTA it launches: at most a few MB). ULY_EINVAL if the plan does not meet
 * the fused call's requirements. */
int ulysses_qk_fused_backward_workspace(ulysses_plan_t plan, size_t* bytes);

/* Size of the scratch array compiled into the library for
 * ulysses_a2a_4d_qk_fused_backward_static: 2 MiB, which holds the dw partial sums of 1,024 CTAs
 * at d = 256 (a GB300 launches at most 608). */
#define ULYSSES_STATIC_SCRATCH_BYTES (2u * 1024u * 1024u)

/*
 * ulysses_a2a_4d_qk_fused_backward without a workspace argument: the same kernels, arguments,
 * results and errors, with the dw partial sums kept in a fixed scratch array inside the library
 * (a file-scope __device__ array of ULYSSES_STATIC_SCRATCH_BYTES). The pages describe no
 * counterpart: it exists for callers that cannot allocate device memory around the call, such as
 * a C caller with no allocator of its own, or code whose device memory is all held by another
 * allocator (a framework's caching pool) or that must not enter an allocator between launches,
 * where cudaMalloc and cudaFree may synchronise the device. The call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library call.
 *   Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, checked) and keeps it; the CUDA runtime may load the library's device
 *   code, array included, at that point (the array is part of the loaded module, not a per-call
 *   allocation). As with the library's other first-call set-up (device attributes, kernel
 *   attributes), make that first call before any stream capture.
 *   Contents: nothing in the array needs to start at zero; every slot the reduction reads is
 *   written in full by the same call's kernel first.
 *   Concurrency: the array is one per device and per process. Calls queued on one stream are
 *   ordered and safe; two calls that may run at the same time on one device (different streams,
 *   or different host threads without ordering) race on it and give wrong dw. Use
 *   ulysses_a2a_4d_qk_fused_backward with separate workspaces for those.
 *   ULY_ESCRATCH when ulysses_qk_fused_backward_workspace for `plan` exceeds
 *   ULYSSES_STATIC_SCRATCH_BYTES (nothing is queued then).
 */
int ulysses_a2a_4d_qk_fused_backward_static(ulysses_plan_t plan, void* const* dq_out,
                                            void* const* dk_out, const void* const* q_in,
                                            const void* const* k_in, const void* const* dq_in,
                                            const void* const* dk_in, const float* rms_w,
                                            float* dw, float eps, float rope_theta, void* stream);

/*
 * The fused call on interleaved packed QKV, the layout a fused QKV projection writes (FastVideo,
 * "Ulysses performance on GB200": packed QKV or QKVG): rank q's input is one (b, s_q, 3, N, d)
 * tensor (bf16 or fp16) whose planes are q, k and v. In one launch per chunk, q and k are normalised,
 * rotated and placed as ulysses_a2a_4d_qk_fused does, and v is placed by mode 0 unchanged
 * (bit-exact).
 *   qkv_in          W device pointers, rank q's (b, s_q, 3, N, d) of the plan's dtype.
 *   q_out, k_out, v_out   W device pointers each, rank r's (b, S, n_r, d), same dtype.
 *   rms_w, eps, rope_theta, plan requirements: as ulysses_a2a_4d_qk_fused. The chunk cap applies
 *   per plane (one launch reads up to three times the cap from a rank).
 */
int ulysses_a2a_4d_qkv_fused(ulysses_plan_t plan, const void* const* qkv_in, void* const* q_out,
                             void* const* k_out, void* const* v_out, const float* rms_w, float eps,
                             float rope_theta, void* stream);

/*
 * The fused call on any packed input of C planes per token (FastVideo, "Ulysses performance on
 * GB200": packed QKV or QKVG, the layouts a fused projection writes): rank q's input holds b * s_q
 * tokens, token (bb, i) starting (bb * s_q + i) * token_pitch bytes in, and within a token plane
 * c's rows (N heads of d elements) start at byte c * N * d * elem_size. In one launch per chunk,
 * the rows of plane q_plane and of plane k_plane are normalised, rotated and placed as
 * ulysses_a2a_4d_qk_fused does (q_plane with rms_w's first row, k_plane with its second), and
 * every other plane is placed by mode 0 unchanged (bit-exact). ulysses_a2a_4d_qkv_fused is the
 * case planes = 3, q_plane = 0, k_plane = 1, token_pitch = 3 * N * d * elem_size.
 *   planes          2 .. 8.
 *   q_plane, k_plane   distinct, in [0, planes).
 *   token_pitch     bytes between consecutive tokens, >= planes * N * d * elem_size, below 2^31
 *                   and a multiple of 16 (ULY_EALIGN otherwise); bytes of a token beyond its planes
 *                   are not read.
 *   packed_in       W device pointers, rank q's b * s_q * token_pitch bytes (plan's dtype).
 *   outs            planes * W device pointers, plane-major: outs[c * W + r] is rank r's
 *                   (b, S, n_r, d) output of plane c.
 *   rms_w, eps, rope_theta, plan requirements: as ulysses_a2a_4d_qk_fused. The chunk cap applies
 *   per plane. Outputs may not overlap inputs or each other (ULY_EOVERLAP).
 */
int ulysses_a2a_4d_packed_fused(ulysses_plan_t plan, int planes, int q_plane, int k_plane,
                                int64_t token_pitch, const void* const* packed_in,
                                void* const* outs, const float* rms_w, float eps, float rope_theta,
                                void* stream);

/*
 * Backward of ulysses_a2a_4d_qkv_fused on the same plan (the pairing of the interleaved call, as
 * ulysses_a2a_4d_qk_fused_backward is of the separate one): the gradient of the packed input
 * (b, s_q, 3, N, d) from the gradients of the three outputs. Planes q and k receive the fused
 * RMSNorm + RoPE vector-Jacobian product exactly as ulysses_a2a_4d_qk_fused_backward computes it;
 * plane v receives the v gradient moved by mode 1 (bit-exact). One launch per chunk covers all
 * three planes, plus the dw reduction.
 *   dqkv_out        W device pointers, rank q's (b, s_q, 3, N, d) of the plan's dtype.
 *   qkv_in          W device pointers, the forward's packed inputs (only planes q and k are read).
 *   dq_in, dk_in, dv_in   W device pointers each, gradients of q_out, k_out, v_out, rank r's
 *                   (b, S, n_r, d).
 *   rms_w, dw, eps, rope_theta, workspace, plan requirements and errors: as
 *   ulysses_a2a_4d_qk_fused_backward (the same workspace size).
 */
int ulysses_a2a_4d_qkv_fused_backward(ulysses_plan_t plan, void* const* dqkv_out,
                                      const void* const* qkv_in, const void* const* dq_in,
                                      const void* const* dk_in, const void* const* dv_in,
                                      const float* rms_w, float* dw, float eps, float rope_theta,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward of ulysses_a2a_4d_packed_fused on the same plan and packing (the general form of
 * ulysses_a2a_4d_qkv_fused_backward, which is its case planes = 3, q_plane = 0, k_plane = 1,
 * token_pitch = 3 * N * d * elem_size): the gradient of the packed input from the gradients of
 * every plane's output. The q and k planes receive the fused RMSNorm + RoPE vector-Jacobian
 * product exactly as ulysses_a2a_4d_qk_fused_backward computes it; every other plane receives its
 * output gradient moved by mode 1 (bit-exact). Bytes of a token beyond its planes are not written.
 * One launch per chunk covers all planes, plus the dw reduction.
 *   planes, q_plane, k_plane, token_pitch   as ulysses_a2a_4d_packed_fused.
 *   dpacked_out     W device pointers, rank q's b * s_q * token_pitch bytes.
 *   packed_in       W device pointers, the forward's packed inputs (only the q and k planes are
 *                   read).
 *   grads           planes * W device pointers, plane-major: grads[c * W + r] is rank r's
 *                   (b, S, n_r, d) gradient of plane c's output.
 *   rms_w, dw, eps, rope_theta, workspace, plan requirements and errors: as
 *   ulysses_a2a_4d_qk_fused_backward (the same workspace size).
 */
int ulysses_a2a_4d_packed_fused_backward(ulysses_plan_t plan, int planes, int q_plane,
                                         int k_plane, int64_t token_pitch,
                                         void* const* dpacked_out, const void* const* packed_in,
                                         const void* const* grads, const float* rms_w, float* dw,
                                         float eps, float rope_theta, void* workspace,
                                         size_t workspace_bytes, void* stream);

/*
 * End-to-end form for host-resident data: copy each rank's input from host_in[k] to dev_in[k],
 * run the relayout, and copy each dev_out[k] back to host_out[k]. The work is cut into about
 * eight ranges of the global sequence (within the chunk cap) so that copies in and copies out
 * overlap: range c is copied in on an auxiliary input stream (after all work queued on `stream`
 * before the call), relaid out on `stream` once its copy in is done, and copied out on an
 * auxiliary output stream while later ranges are copied in; `stream` finally waits for the
 * output stream, so the call is
 * ordered on `stream` as a whole (when `stream` has completed, host_out holds the result). The
 * auxiliary streams and a few events are created once per device on the first such call (no
 * device memory) and reused; concurrent calls from several host threads are serialised while
 * they enqueue. Host buffers should be page-locked for the copies to be asynchronous. Device
 * buffers are the caller's, as above.
 */
int ulysses_a2a_4d_host(ulysses_plan_t plan, int mode, const void* const* host_in,
                        void* const* host_out, void* const* dev_in, void* const* dev_out,
                        void* stream);

/*
 * End-to-end form of ulysses_a2a_4d_qk_fused for host-resident q and k: copy each rank's q and k
 * from host to the device buffers, run the fused call, and copy q_out and k_out back to the
 * host, chunked and overlapped exactly as ulysses_a2a_4d_host. Same arguments and rules as the
 * device form, plus the host buffers.
 */
int ulysses_a2a_4d_qk_fused_host(ulysses_plan_t plan, const void* const* q_host_in,
                                 const void* const* k_host_in, void* const* q_host_out,
                                 void* const* k_host_out, void* const* q_in, void* const* k_in,
                                 void* const* q_out, void* const* k_out, const float* rms_w,
                                 float eps, float rope_theta, void* stream);

/* Synchronise the current device, then return in *status the device status word accumulated by
 * this library's kernels since the last call (0 = no kernel timed out) and clear it. Returns
 * ULY_EDEVICE when the word was non-zero. Bits: 1 (a pipeline wait gave up after 2 s: the
 * outputs of the calls since the last check are incomplete; discard them), 2 (a kernel gave up
 * waiting for its own bulk copies into shared memory before exiting: such a copy never completed,
 * so it may still land in shared memory a later kernel owns; discard the outputs and treat the
 * CUDA context as suspect, i.e. reset it with cudaDeviceReset before further work). Neither bit
 * is set unless the hardware stalls for seconds. */
int ulysses_device_status(unsigned* status);

/*
 * Self-test of the failure path (no counterpart on the pages, which describe hangs on misuse but
 * no detection): queue on `stream` a one-warp kernel that waits on a barrier nothing arrives on,
 * with a limit of limit_us microseconds (1 .. 1,000,000) instead of the kernels' 2 s. The wait
 * gives up, sets the timeout bit (1) of the device status word, and the kernel returns normally,
 * so the context stays usable; ulysses_device_status() then reports ULY_EDEVICE with status 1.
 */
int ulysses_selftest_wait_timeout(unsigned limit_us, void* stream);

/* The cudaError_t value of the last ULY_ECUDA returned on this host thread (0 if none). */
int ulysses_last_cuda_error(void);

/* A static, human-readable name for a status code. */
const char* ulysses_strerror(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int ulysses_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ULYSSES_H */
