// api.cu -- the extern "C" entry points declared in include/ulysses.h: argument checks, chunking,
// argument blocks, launches. All device work goes to the caller's stream; nothing synchronises
// except ulysses_device_status().
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <atomic>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/ulysses.h"
#include "plan.h"
#include "tensor_map.h"

namespace uly {
int64_t relayout_unit_bytes(int engine);
cudaError_t relayout_launch(const RelayoutArgs& a, int mode, int engine, cudaStream_t stream,
                            int device, int sm_count, int64_t max_grid);
cudaError_t relayout_status(unsigned* status, bool clear);
bool relayout_tensor_fits(const Plan& p);
bool relayout_tensor_preferred(const Plan& p, int sm_count);
cudaError_t relayout_tensor_launch(const Plan& p, const ChunkRows& rows, uint8_t* const* seq,
                                   uint8_t* const* head, int mode, cudaStream_t stream, int device,
                                   int sm_count, int64_t max_grid);
RowRing relayout_row_ring(const Plan& p, int mode);
int64_t relayout_tile_rows(int64_t row_bytes, int64_t stage_bytes);
cudaError_t relayout_rows_launch(const RowTileArgs& a, int mode, const RowRing& ring,
                                 cudaStream_t stream, int device, int sm_count, int64_t max_grid);
void fused_geometry(const Plan& p, int planes, int64_t* tokens_per_unit, int* stages,
                    uint32_t* stage_bytes, int* ctas_per_sm);
cudaError_t fused_launch(const FusedArgs& a, cudaStream_t stream, int device, int sm_count,
                         int64_t max_grid);
cudaError_t fused_status(unsigned* status, bool clear);
bool fused_tensor_fits(const Plan& p);
bool fused_tensor_preferred(const Plan& p);
cudaError_t fused_tensor_launch(const Plan& p, const FusedArgs& f, const ChunkRows& rows,
                                cudaStream_t stream, int device, int sm_count, int64_t max_grid);
cudaError_t fused_tensor_status(unsigned* status, bool clear);
bool fused_bwd_group_major_preferred(const Plan& p);
void fused_bwd_geometry(const Plan& p, bool group_major, int64_t* tokens_per_unit, int* stages,
                        uint32_t* stage_bytes, int* ctas_per_sm);
int64_t fused_bwd_grid(const FusedBwdArgs& a, int sm_count, int64_t max_grid);
cudaError_t fused_bwd_launch(const FusedBwdArgs& a, float* dw, bool accumulate, cudaStream_t stream,
                             int device, int sm_count, int64_t max_grid);
cudaError_t fused_bwd_status(unsigned* status, bool clear);
cudaError_t selftest_timeout_launch(uint64_t limit_ns, cudaStream_t stream);
}  // namespace uly

using namespace uly;

namespace {

thread_local int t_last_cuda_error = 0;

int cuda_fail(cudaError_t e)
{
    t_last_cuda_error = int(e);
    return ULY_ECUDA;
}

struct DeviceInfo {
    int device;
    int sm_count;
};

int current_device(DeviceInfo* info)
{
    static std::atomic<int> sm_counts[64];  // per device, filled on first use by any thread
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= 64) return ULY_EINVAL;
    int sms = sm_counts[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        sm_counts[dev].store(sms, std::memory_order_relaxed);
    }
    info->device = dev;
    info->sm_count = sms;
    return ULY_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks W pointers against their sizes: present when non-empty, 16-byte aligned.
int check_ptrs(const void* const* ptrs, const int64_t* bytes, int W)
{
    if (!ptrs) return ULY_EINVAL;
    for (int k = 0; k < W; ++k) {
        if (bytes[k] == 0) continue;
        if (!ptrs[k]) return ULY_EINVAL;
        if (!aligned16(ptrs[k])) return ULY_EALIGN;
    }
    return ULY_OK;
}

bool ranges_overlap(const void* a, int64_t na, const void* b, int64_t nb)
{
    if (na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + uintptr_t(nb) && b0 < a0 + uintptr_t(na);
}

// Outputs may overlap neither inputs nor each other (inputs may alias each other: they are read).
int check_overlap(const void* const* in, const int64_t* in_bytes, int n_in, const void* const* out,
                  const int64_t* out_bytes, int n_out)
{
    for (int o = 0; o < n_out; ++o) {
        for (int i = 0; i < n_in; ++i)
            if (ranges_overlap(out[o], out_bytes[o], in[i], in_bytes[i])) return ULY_EOVERLAP;
        for (int o2 = o + 1; o2 < n_out; ++o2)
            if (ranges_overlap(out[o], out_bytes[o], out[o2], out_bytes[o2])) return ULY_EOVERLAP;
    }
    return ULY_OK;
}

void side_bytes(const Plan& p, int mode, int64_t* in_b, int64_t* out_b)
{
    for (int k = 0; k < p.W; ++k) {
        const int64_t sq = seq_side_bytes(p, k), hd = head_side_bytes(p, k);
        in_b[k] = mode == 0 ? sq : hd;
        out_b[k] = mode == 0 ? hd : sq;
    }
}

// Argument checks of a relayout call (no CUDA call).
int relayout_check(const Plan& p, int mode, int engine, const void* const* in_ptrs,
                   void* const* out_ptrs)
{
    if (mode != 0 && mode != 1) return ULY_EINVAL;
    if (engine != ULY_ENGINE_AUTO && engine != ULY_ENGINE_TMA && engine != ULY_ENGINE_VEC &&
        engine != ULY_ENGINE_CE && engine != ULY_ENGINE_TENSOR)
        return ULY_EINVAL;
    int64_t in_b[kMaxW], out_b[kMaxW];
    side_bytes(p, mode, in_b, out_b);
    int rc = check_ptrs(in_ptrs, in_b, p.W);
    if (rc) return rc;
    rc = check_ptrs(const_cast<const void* const*>(out_ptrs), out_b, p.W);
    if (rc) return rc;
    return check_overlap(in_ptrs, in_b, p.W, const_cast<const void* const*>(out_ptrs), out_b, p.W);
}

// The copy-engine form of one chunk: per (source shard q, destination rank r, batch index) one
// pitched 2D copy of the chunk's rows of shard q: n_r * d * e bytes wide, the row pitch N * d * e
// on the sequence side and n_r * d * e on the head side (the pages' design, pitched copies on the
// copy engines, here between buffers of one GPU).
int relayout_rows_ce(const Plan& p, int mode, const void* const* in_ptrs, void* const* out_ptrs,
                     const ChunkRows& rows, cudaStream_t stream)
{
    const int64_t elem_row = p.d * p.e;  // bytes of one head row
    for (int q = 0; q < p.W; ++q) {
        const int64_t cnt = rows.cnt[q];
        if (cnt == 0) continue;
        for (int r = 0; r < p.W; ++r) {
            const int64_t width = p.n[r] * elem_row;
            if (width == 0) continue;
            for (int64_t bb = 0; bb < p.b; ++bb) {
                uint8_t* seq = static_cast<uint8_t*>(mode == 0 ? const_cast<void*>(in_ptrs[q])
                                                               : out_ptrs[q]) +
                               ((bb * p.s[q] + rows.lo[q]) * p.N + p.head_off[r]) * elem_row;
                uint8_t* head = static_cast<uint8_t*>(mode == 0 ? out_ptrs[r]
                                                                : const_cast<void*>(in_ptrs[r])) +
                                (bb * p.S + p.seq_off[q] + rows.lo[q]) * width;
                const size_t seq_pitch = size_t(p.N * elem_row), head_pitch = size_t(width);
                cudaError_t e = mode == 0
                    ? cudaMemcpy2DAsync(head, head_pitch, seq, seq_pitch, size_t(width), size_t(cnt),
                                        cudaMemcpyDeviceToDevice, stream)
                    : cudaMemcpy2DAsync(seq, seq_pitch, head, head_pitch, size_t(width), size_t(cnt),
                                        cudaMemcpyDeviceToDevice, stream);
                if (e != cudaSuccess) return cuda_fail(e);
            }
        }
    }
    return ULY_OK;
}

// One launch of the relayout over the given rows of every sequence shard.
int relayout_rows(const Plan& p, int mode, int engine, const void* const* in_ptrs,
                  void* const* out_ptrs, const ChunkRows& rows, cudaStream_t stream,
                  const DeviceInfo& dev)
{
    if (engine == ULY_ENGINE_AUTO)
        engine = relayout_tensor_preferred(p, dev.sm_count) ? ULY_ENGINE_TENSOR : ULY_ENGINE_TMA;
    if (engine == ULY_ENGINE_CE) return relayout_rows_ce(p, mode, in_ptrs, out_ptrs, rows, stream);
    uint8_t* seq[kMaxW];
    uint8_t* head[kMaxW];
    for (int k = 0; k < p.W; ++k) {
        uint8_t* in = static_cast<uint8_t*>(const_cast<void*>(in_ptrs[k]));
        uint8_t* out = static_cast<uint8_t*>(out_ptrs[k]);
        seq[k] = mode == 0 ? in : out;
        head[k] = mode == 0 ? out : in;
    }
    if (engine == ULY_ENGINE_TENSOR) {  // one tensor-map box per unit; runs over 2 KiB: TMA
        if (relayout_tensor_fits(p)) {
            cudaError_t e = relayout_tensor_launch(p, rows, seq, head, mode, stream, dev.device,
                                                   dev.sm_count, p.max_ctas);
            return e == cudaSuccess ? ULY_OK : cuda_fail(e);
        }
        engine = ULY_ENGINE_TMA;
    }
    // TMA engine: whole-row tiles when a row fits a stage, row-run segments otherwise
    const RowRing ring = relayout_row_ring(p, mode);
    const int64_t tile_rows =
        engine == ULY_ENGINE_TMA ? relayout_tile_rows(p.N * p.d * p.e, ring.stage_bytes) : 0;
    cudaError_t e;
    if (tile_rows > 0) {
        RowTileArgs t;
        std::memset(&t, 0, sizeof t);
        for (int k = 0; k < p.W; ++k) {
            t.seq_ptr[k] = seq[k];
            t.head_ptr[k] = head[k];
        }
        build_row_tiles(p, rows, tile_rows, &t);
        t.stage_bytes = ring.stage_bytes;
        e = relayout_rows_launch(t, mode, ring, stream, dev.device, dev.sm_count, p.max_ctas);
    } else {
        RelayoutArgs a;
        std::memset(&a, 0, sizeof a);
        for (int k = 0; k < p.W; ++k) {
            a.seq_ptr[k] = seq[k];
            a.head_ptr[k] = head[k];
        }
        build_relayout_units(p, rows, relayout_unit_bytes(engine), &a);
        e = relayout_launch(a, mode, engine, stream, dev.device, dev.sm_count, p.max_ctas);
    }
    return e == cudaSuccess ? ULY_OK : cuda_fail(e);
}

int relayout_impl(const Plan& p, int mode, int engine, const void* const* in_ptrs,
                  void* const* out_ptrs, cudaStream_t stream)
{
    int rc = relayout_check(p, mode, engine, in_ptrs, out_ptrs);
    if (rc) return rc;
    int64_t C = 0;
    if ((rc = num_chunks(p, &C))) return rc;
    DeviceInfo dev;
    if ((rc = current_device(&dev))) return rc;
    for (int64_t c = 0; c < C; ++c) {
        ChunkRows rows;
        chunk_rows(p, C, c, &rows);
        if ((rc = relayout_rows(p, mode, engine, in_ptrs, out_ptrs, rows, stream, dev))) return rc;
    }
    return ULY_OK;
}

// A packed fused input: rank q's b * s_q tokens, `pitch` bytes apart, each holding `planes` planes
// of N * d elements (plane c at byte c * N * d * e of the token); outs[c * W + r] is rank r's
// (b, S, n_r, d) output of plane c (q_plane's and k_plane's receive the transformed rows).
struct PackedIn {
    const void* const* in;
    int planes, q_plane, k_plane;
    int64_t pitch;
    void* const* outs;
};

// Head dimensions of the fused calls: every multiple of 8 from 8 to 256 (a head row of 2-byte
// elements is then a whole number of 16-byte words). Powers of two run kernels compiled for
// their d; the others the same kernels with d read at run time (fused_row.cuh).
bool fused_head_dim_ok(int64_t d) { return d >= 8 && d <= kMaxFusedD && d % 8 == 0; }

// Checks of a fused call (no CUDA call) and its argument block, without the unit tables. Either
// q_in, k_in, q_out and k_out are given (separate tensors) or a packed input (pk).
int fused_prepare(const Plan& p, const void* const* q_in, const void* const* k_in,
                  void* const* q_out, void* const* k_out, const PackedIn* pk, const float* rms_w,
                  float eps, float rope_theta, FusedArgs* a, int64_t* tokens_per_unit)
{
    if (p.dtype != ULY_BF16 && p.dtype != ULY_F16) return ULY_EINVAL;
    if (!fused_head_dim_ok(p.d)) return ULY_EINVAL;
    if (p.S >= (int64_t(1) << 24)) return ULY_EINVAL;  // positions must be exact in fp32
    if (!(eps >= 0.0f) || !(rope_theta > 0.0f)) return ULY_EINVAL;
    if (!rms_w) return ULY_EINVAL;
    if (!aligned16(rms_w)) return ULY_EALIGN;
    const int W = p.W;
    const int64_t row_bytes = p.N * p.d * p.e;
    int64_t in_b[kMaxW], out_b[kMaxW], packed_b[kMaxW];
    side_bytes(p, 0, in_b, out_b);
    if (pk) {
        if (!pk->in || !pk->outs || pk->planes < 2 || pk->planes > kMaxPlanes ||
            pk->q_plane < 0 || pk->q_plane >= pk->planes || pk->k_plane < 0 ||
            pk->k_plane >= pk->planes || pk->q_plane == pk->k_plane ||
            pk->pitch < pk->planes * row_bytes || pk->pitch >= (int64_t(1) << 31))
            return ULY_EINVAL;
        if (pk->pitch % 16 != 0) return ULY_EALIGN;
        for (int k = 0; k < W; ++k) {
            if (p.b * p.s[k] > INT64_MAX / pk->pitch) return ULY_EINVAL;  // bytes overflow
            packed_b[k] = p.b * p.s[k] * pk->pitch;
        }
        q_out = pk->outs + size_t(pk->q_plane) * W;
        k_out = pk->outs + size_t(pk->k_plane) * W;
    }
    int rc;
    if (pk) {
        if ((rc = check_ptrs(pk->in, packed_b, W))) return rc;
        for (int c = 0; c < pk->planes; ++c)
            if ((rc = check_ptrs(const_cast<const void* const*>(pk->outs + size_t(c) * W), out_b, W)))
                return rc;
    } else if ((rc = check_ptrs(q_in, in_b, W)) || (rc = check_ptrs(k_in, in_b, W)) ||
               (rc = check_ptrs(const_cast<const void* const*>(q_out), out_b, W)) ||
               (rc = check_ptrs(const_cast<const void* const*>(k_out), out_b, W))) {
        return rc;
    }
    // every input (plus the weights) against every output
    const void* ins[2 * kMaxW + 1];
    int64_t ins_b[2 * kMaxW + 1];
    const void* outs[kMaxPlanes * kMaxW];
    int64_t outs_b[kMaxPlanes * kMaxW];
    int n_in = 0, n_out = 0;
    for (int k = 0; k < W; ++k) {
        if (pk) {
            ins[n_in] = pk->in[k];
            ins_b[n_in++] = packed_b[k];
            for (int c = 0; c < pk->planes; ++c) {
                outs[n_out] = pk->outs[size_t(c) * W + k];
                outs_b[n_out++] = out_b[k];
            }
        } else {
            ins[n_in] = q_in[k];
            ins_b[n_in++] = in_b[k];
            ins[n_in] = k_in[k];
            ins_b[n_in++] = in_b[k];
            outs[n_out] = q_out[k];
            outs_b[n_out++] = out_b[k];
            outs[n_out] = k_out[k];
            outs_b[n_out++] = out_b[k];
        }
    }
    ins[n_in] = rms_w;
    ins_b[n_in++] = 2 * p.d * int64_t(sizeof(float));
    if ((rc = check_overlap(ins, ins_b, n_in, outs, outs_b, n_out))) return rc;
    int stages = 0, ctas_per_sm = 1;
    uint32_t stage_bytes = 0;
    // a stage holds the q and k rows of tokens_per_unit tokens (a packed call's other-plane units
    // hold one plane's rows of twice as many tokens: the same bytes)
    fused_geometry(p, 2, tokens_per_unit, &stages, &stage_bytes, &ctas_per_sm);
    if (stages == 0) return ULY_EINVAL;  // one token's rows do not fit the stages
    std::memset(a, 0, sizeof *a);
    a->ctas_per_sm = ctas_per_sm;
    a->interleaved = pk ? 1 : 0;
    a->elem_f16 = p.dtype == ULY_F16 ? 1 : 0;
    a->rope_half = p.rope_half;
    if (pk) {
        a->planes = pk->planes;
        a->q_plane = pk->q_plane;
        a->k_plane = pk->k_plane;
        a->tok_pitch = pk->pitch;
        int n_plain = 0;
        for (int c = 0; c < pk->planes; ++c) {
            if (c != pk->q_plane && c != pk->k_plane) a->plain_plane[n_plain++] = c;
            for (int k = 0; k < W; ++k)
                a->plane_out[c][k] = static_cast<uint8_t*>(pk->outs[size_t(c) * W + k]);
        }
    }
    for (int k = 0; k < W; ++k) {
        if (pk) {
            a->packed_in[k] = static_cast<const uint8_t*>(pk->in[k]);
        } else {
            a->q_in[k] = static_cast<const uint8_t*>(q_in[k]);
            a->k_in[k] = static_cast<const uint8_t*>(k_in[k]);
        }
        a->q_out[k] = static_cast<uint8_t*>(q_out[k]);
        a->k_out[k] = static_cast<uint8_t*>(k_out[k]);
    }
    a->rms_w = rms_w;
    a->eps = eps;
    a->stages = stages;
    a->stage_bytes = stage_bytes;
    rope_turns(p.d, double(rope_theta), a->turn_hi, a->turn_lo);
    return ULY_OK;
}

// Whether a fused forward call (separate or packed inputs) takes the row-block tensor-map kernel.
static bool fused_uses_tensor(const Plan& p)
{
    if (p.fused_engine == ULY_ENGINE_TMA || !fused_tensor_fits(p)) return false;
    return p.fused_engine == ULY_ENGINE_TENSOR || fused_tensor_preferred(p);
}

// Whether the backward of the fused call takes row blocks grouped by head group: under the
// plan's fused-kernel setting, where they fit, and under the automatic choice where measured faster.
static bool fused_bwd_uses_group_major(const Plan& p)
{
    if (p.fused_engine == ULY_ENGINE_TMA || !fused_tensor_fits(p)) return false;
    return p.fused_engine == ULY_ENGINE_TENSOR || fused_bwd_group_major_preferred(p);
}

// One launch of the fused kernel over the given rows of every sequence shard.
int fused_rows(const Plan& p, FusedArgs* a, int64_t tokens_per_unit, const ChunkRows& rows,
               cudaStream_t stream, const DeviceInfo& dev)
{
    if (fused_uses_tensor(p)) {
        cudaError_t e = fused_tensor_launch(p, *a, rows, stream, dev.device, dev.sm_count, p.max_ctas);
        return e == cudaSuccess ? ULY_OK : cuda_fail(e);
    }
    if (a->interleaved)
        build_fused_units(p, rows, tokens_per_unit, 2 * tokens_per_unit, a->planes, a);
    else
        build_fused_units(p, rows, tokens_per_unit, tokens_per_unit, 1, a);
    cudaError_t e = fused_launch(*a, stream, dev.device, dev.sm_count, p.max_ctas);
    return e == cudaSuccess ? ULY_OK : cuda_fail(e);
}

// The device forms of the fused calls: checks, then one launch per chunk of the plan.
int fused_device(const Plan& p, const void* const* q_in, const void* const* k_in,
                 void* const* q_out, void* const* k_out, const PackedIn* pk, const float* rms_w,
                 float eps, float rope_theta, cudaStream_t stream)
{
    FusedArgs a;
    int64_t T = 0;
    int rc = fused_prepare(p, q_in, k_in, q_out, k_out, pk, rms_w, eps, rope_theta, &a, &T);
    if (rc) return rc;
    int64_t C = 0;
    if ((rc = num_chunks(p, &C))) return rc;
    DeviceInfo dev;
    if ((rc = current_device(&dev))) return rc;
    for (int64_t c = 0; c < C; ++c) {
        ChunkRows rows;
        chunk_rows(p, C, c, &rows);
        if ((rc = fused_rows(p, &a, T, rows, stream, dev))) return rc;
    }
    return ULY_OK;
}

// ---- backward of the fused QK call -------------------------------------------------------------
// Plan requirements (as the forward), geometry, and the partial-sum bytes for the device the
// caller is on: one 2 x d fp32 slot per CTA of the largest launch.
int fused_bwd_setup(const Plan& p, const DeviceInfo& dev, int64_t* tokens_per_unit, int* stages,
                    uint32_t* stage_bytes, int* ctas_per_sm, size_t* workspace_bytes)
{
    if (p.dtype != ULY_BF16 && p.dtype != ULY_F16) return ULY_EINVAL;
    if (!fused_head_dim_ok(p.d)) return ULY_EINVAL;
    if (p.S >= (int64_t(1) << 24)) return ULY_EINVAL;  // positions must be exact in fp32
    fused_bwd_geometry(p, fused_bwd_uses_group_major(p), tokens_per_unit, stages, stage_bytes,
                       ctas_per_sm);
    if (*stages == 0) return ULY_EINVAL;  // one token's rows do not fit the stages
    *workspace_bytes = size_t(dev.sm_count) * size_t(*ctas_per_sm) * size_t(2 * p.d) * sizeof(float);
    return ULY_OK;
}

// The launches of a backward whose pointers, tensor count and token stride are set in `a`.
int fused_bwd_run(const Plan& p, FusedBwdArgs& a, const DeviceInfo& dev, int64_t T, int stages,
                  uint32_t stage_bytes, int ctas_per_sm, const float* rms_w, float* dw, float eps,
                  float rope_theta, void* workspace, cudaStream_t stream)
{
    int64_t C = 0;
    int rc = num_chunks(p, &C);
    if (rc) return rc;
    a.rms_w = rms_w;
    a.dw_part = static_cast<float*>(workspace);
    a.elem_f16 = p.dtype == ULY_F16 ? 1 : 0;
    a.rope_half = p.rope_half;
    a.eps = eps;
    a.stages = stages;
    a.stage_bytes = stage_bytes;
    a.ctas_per_sm = ctas_per_sm;
    a.group_major = fused_bwd_uses_group_major(p) ? 1 : 0;  // the same choice as the geometry's
    a.n_eq = int32_t(p.n[0]);
    a.run = uint32_t(p.n[0] * p.d * p.e);
    rope_turns(p.d, double(rope_theta), a.turn_hi, a.turn_lo);
    for (int64_t c = 0; c < C; ++c) {
        ChunkRows rows;
        chunk_rows(p, C, c, &rows);
        build_fused_bwd_units(p, rows, T, &a);
        if (a.group_major) {  // maps of this launch's rows: the forward inputs, and the other
                              // planes' gradient outputs of a packed call
            for (int t = 0; t < a.tensors; ++t) {
                for (int q = 0; q < p.W; ++q) {
                    if (rows.cnt[q] == 0) continue;
                    CUtensorMap* map = t < 2 ? &a.xmap[t][q] : &a.dmap[t - 2][q];
                    const uint8_t* base = t < 2 ? a.x_in[t][q] : a.dx_out[t][q];
                    if (!encode_group_map(map, base + rows.lo[q] * a.tok_stride, a.run,
                                          rows.cnt[q], p.W, p.b, a.tok_stride,
                                          p.s[q] * a.tok_stride, T))
                        return cuda_fail(cudaErrorInvalidValue);
                }
            }
        }
        cudaError_t e = fused_bwd_launch(a, dw, c > 0, stream, dev.device, dev.sm_count, p.max_ctas);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return ULY_OK;
}

// Checks shared by both backward forms: plan, scalars, weights, dw and workspace.
int fused_bwd_common(const Plan& p, const DeviceInfo& dev, const float* rms_w, float* dw,
                     float eps, float rope_theta, void* workspace, size_t workspace_bytes,
                     int64_t* T, int* stages, uint32_t* stage_bytes, int* ctas_per_sm, size_t* need)
{
    int rc = fused_bwd_setup(p, dev, T, stages, stage_bytes, ctas_per_sm, need);
    if (rc) return rc;
    if (!(eps >= 0.0f) || !(rope_theta > 0.0f)) return ULY_EINVAL;
    if (!rms_w || !dw || !workspace || workspace_bytes < *need) return ULY_EINVAL;
    if (!aligned16(rms_w) || !aligned16(dw) || !aligned16(workspace)) return ULY_EALIGN;
    return ULY_OK;
}

int fused_bwd_device(const Plan& p, void* const* dq_out, void* const* dk_out,
                     const void* const* q_in, const void* const* k_in, const void* const* dq_in,
                     const void* const* dk_in, const float* rms_w, float* dw, float eps,
                     float rope_theta, void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    int64_t T = 0;
    int stages = 0, ctas_per_sm = 1;
    uint32_t stage_bytes = 0;
    size_t need = 0;
    if ((rc = fused_bwd_common(p, dev, rms_w, dw, eps, rope_theta, workspace, workspace_bytes, &T,
                               &stages, &stage_bytes, &ctas_per_sm, &need)))
        return rc;
    int64_t seq_b[kMaxW], head_b[kMaxW];
    side_bytes(p, 0, seq_b, head_b);
    if ((rc = check_ptrs(q_in, seq_b, p.W)) || (rc = check_ptrs(k_in, seq_b, p.W)) ||
        (rc = check_ptrs(dq_in, head_b, p.W)) || (rc = check_ptrs(dk_in, head_b, p.W)) ||
        (rc = check_ptrs(const_cast<const void* const*>(dq_out), seq_b, p.W)) ||
        (rc = check_ptrs(const_cast<const void* const*>(dk_out), seq_b, p.W)))
        return rc;
    // every input (plus the weights) against every output (plus dw and the workspace)
    const void* ins[4 * kMaxW + 1];
    int64_t ins_b[4 * kMaxW + 1];
    const void* outs[2 * kMaxW + 2];
    int64_t outs_b[2 * kMaxW + 2];
    int n_in = 0, n_out = 0;
    for (int k = 0; k < p.W; ++k) {
        ins[n_in] = q_in[k];
        ins_b[n_in++] = seq_b[k];
        ins[n_in] = k_in[k];
        ins_b[n_in++] = seq_b[k];
        ins[n_in] = dq_in[k];
        ins_b[n_in++] = head_b[k];
        ins[n_in] = dk_in[k];
        ins_b[n_in++] = head_b[k];
        outs[n_out] = dq_out[k];
        outs_b[n_out++] = seq_b[k];
        outs[n_out] = dk_out[k];
        outs_b[n_out++] = seq_b[k];
    }
    ins[n_in] = rms_w;
    ins_b[n_in++] = 2 * p.d * int64_t(sizeof(float));
    outs[n_out] = dw;
    outs_b[n_out++] = 2 * p.d * int64_t(sizeof(float));
    outs[n_out] = workspace;
    outs_b[n_out++] = int64_t(need);
    if ((rc = check_overlap(ins, ins_b, n_in, outs, outs_b, n_out))) return rc;
    FusedBwdArgs a;
    std::memset(&a, 0, sizeof a);
    for (int k = 0; k < p.W; ++k) {
        a.x_in[0][k] = static_cast<const uint8_t*>(q_in[k]);
        a.x_in[1][k] = static_cast<const uint8_t*>(k_in[k]);
        a.g_in[0][k] = static_cast<const uint8_t*>(dq_in[k]);
        a.g_in[1][k] = static_cast<const uint8_t*>(dk_in[k]);
        a.dx_out[0][k] = static_cast<uint8_t*>(dq_out[k]);
        a.dx_out[1][k] = static_cast<uint8_t*>(dk_out[k]);
    }
    a.tensors = 2;
    a.tok_stride = int32_t(p.N * p.d * p.e);
    return fused_bwd_run(p, a, dev, T, stages, stage_bytes, ctas_per_sm, rms_w, dw, eps,
                         rope_theta, workspace, stream);
}

// The backward of a packed fused call: for the q and k planes the fused VJP, for every other plane
// its gradient by mode 1, all written into rank q's packed gradient (the same pitch; a token's
// columns beyond its planes are not written). grads[c * W + r] is rank r's gradient of plane c's
// output.
int packed_bwd_device(const Plan& p, void* const* dpacked_out, const void* const* packed_in,
                      int planes, int q_plane, int k_plane, int64_t pitch,
                      const void* const* grads, const float* rms_w, float* dw, float eps,
                      float rope_theta, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream)
{
    const int W = p.W;
    const int64_t row = p.N * p.d * p.e;  // one token's heads of one plane
    if (!dpacked_out || !packed_in || !grads || planes < 2 || planes > kMaxPlanes ||
        q_plane < 0 || q_plane >= planes || k_plane < 0 || k_plane >= planes ||
        q_plane == k_plane || pitch < planes * row || pitch >= (int64_t(1) << 31))
        return ULY_EINVAL;
    if (pitch % 16 != 0) return ULY_EALIGN;
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    int64_t T = 0;
    int stages = 0, ctas_per_sm = 1;
    uint32_t stage_bytes = 0;
    size_t need = 0;
    if ((rc = fused_bwd_common(p, dev, rms_w, dw, eps, rope_theta, workspace, workspace_bytes, &T,
                               &stages, &stage_bytes, &ctas_per_sm, &need)))
        return rc;
    int64_t seq_b[kMaxW], head_b[kMaxW], packed_b[kMaxW];
    side_bytes(p, 0, seq_b, head_b);
    for (int k = 0; k < W; ++k) {
        if (p.b * p.s[k] > INT64_MAX / pitch) return ULY_EINVAL;  // bytes overflow
        packed_b[k] = p.b * p.s[k] * pitch;
    }
    if ((rc = check_ptrs(packed_in, packed_b, W)) ||
        (rc = check_ptrs(const_cast<const void* const*>(dpacked_out), packed_b, W)))
        return rc;
    for (int c = 0; c < planes; ++c)
        if ((rc = check_ptrs(grads + size_t(c) * W, head_b, W))) return rc;
    const void* ins[(kMaxPlanes + 1) * kMaxW + 1];
    int64_t ins_b[(kMaxPlanes + 1) * kMaxW + 1];
    const void* outs[kMaxW + 2];
    int64_t outs_b[kMaxW + 2];
    int n_in = 0, n_out = 0;
    for (int k = 0; k < W; ++k) {
        ins[n_in] = packed_in[k];
        ins_b[n_in++] = packed_b[k];
        for (int c = 0; c < planes; ++c) {
            ins[n_in] = grads[size_t(c) * W + k];
            ins_b[n_in++] = head_b[k];
        }
        outs[n_out] = dpacked_out[k];
        outs_b[n_out++] = packed_b[k];
    }
    ins[n_in] = rms_w;
    ins_b[n_in++] = 2 * p.d * int64_t(sizeof(float));
    outs[n_out] = dw;
    outs_b[n_out++] = 2 * p.d * int64_t(sizeof(float));
    outs[n_out] = workspace;
    outs_b[n_out++] = int64_t(need);
    if ((rc = check_overlap(ins, ins_b, n_in, outs, outs_b, n_out))) return rc;
    // tensor t of the kernel: 0 the q plane, 1 the k plane, 2 .. the other planes in order
    int plane_of[kMaxPlanes];
    plane_of[0] = q_plane;
    plane_of[1] = k_plane;
    for (int c = 0, t = 2; c < planes; ++c)
        if (c != q_plane && c != k_plane) plane_of[t++] = c;
    FusedBwdArgs a;
    std::memset(&a, 0, sizeof a);
    for (int k = 0; k < W; ++k) {
        const uint8_t* in = static_cast<const uint8_t*>(packed_in[k]);
        uint8_t* out = static_cast<uint8_t*>(dpacked_out[k]);
        for (int t = 0; t < planes; ++t) {
            const int64_t off = int64_t(plane_of[t]) * row;
            if (t < 2) a.x_in[t][k] = in ? in + off : nullptr;
            a.dx_out[t][k] = out ? out + off : nullptr;
            a.g_in[t][k] = static_cast<const uint8_t*>(grads[size_t(plane_of[t]) * W + k]);
        }
    }
    a.tensors = planes;
    a.tok_stride = int32_t(pitch);
    return fused_bwd_run(p, a, dev, T, stages, stage_bytes, ctas_per_sm, rms_w, dw, eps,
                         rope_theta, workspace, stream);
}

// ---- backward with library-owned scratch ----------------------------------------------------------
// The dw partial sums of ulysses_a2a_4d_qk_fused_backward_static live in this array; its device
// address is looked up once per device and kept. No part of it needs initial contents: each
// launch's CTAs write their slots in full before the reduction reads them.
static __device__ __align__(256) float g_static_scratch[ULYSSES_STATIC_SCRATCH_BYTES / sizeof(float)];

std::mutex g_scratch_mu;
void* g_scratch_addr[64];

int static_scratch(int device, void** out)
{
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[device]) {
        void* addr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&addr, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        if (!addr || !aligned16(addr)) return ULY_EALIGN;
        g_scratch_addr[device] = addr;
    }
    *out = g_scratch_addr[device];
    return ULY_OK;
}

// ---- host-buffer entry points: chunked copy-in / kernel / copy-out pipeline ---------------------
// Host<->device copies run on the copy engines in both directions at once, so the call is cut
// into sequence chunks and run as a three-stream pipeline: chunk c's inputs are copied in on an
// input stream (which first waits for everything already queued on the caller's stream), chunk c
// is relaid out on the caller's stream once its copy-in is done, and an output stream copies its
// results back once its kernel is done. So copies in follow one another without waiting for the
// kernels, and chunk c is copied out while later chunks are copied in. The caller's stream finally
// waits for the output stream, so from the caller's side the whole call is ordered on its stream
// like any other. The streams and events are created once per device, on first use, and reused;
// a mutex serialises the enqueueing of concurrent calls.
constexpr int kPipeEvents = 4;
#ifndef ULY_HOST_CHUNKS
#define ULY_HOST_CHUNKS 8
#endif
constexpr int64_t kPipeChunks = ULY_HOST_CHUNKS;

struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr;   // copies in
    cudaStream_t aux = nullptr;  // copies out
    cudaEvent_t entry = nullptr;  // the caller's stream when the call was made
    cudaEvent_t in_done[kPipeEvents] = {};
    cudaEvent_t chunk_done[kPipeEvents] = {};
    cudaEvent_t copied_out = nullptr;
};

std::mutex g_pipe_mu;
HostPipe g_pipe[64];

int host_pipe(int device, HostPipe** out)  // caller holds g_pipe_mu
{
    HostPipe& hp = g_pipe[device];
    if (!hp.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&hp.aux, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking);
        for (int i = 0; e == cudaSuccess && i < kPipeEvents; ++i) {
            e = cudaEventCreateWithFlags(&hp.chunk_done[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.in_done[i], cudaEventDisableTiming);
        }
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.copied_out, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.entry, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e);
        hp.ready = true;
    }
    *out = &hp;
    return ULY_OK;
}

// Rows [lo_q, lo_q + cnt_q) of every rank's sequence-side tensor (b, s_q, N, d), per batch index.
cudaError_t copy_seq_rows(const Plan& p, const ChunkRows& rows, void* const* dst,
                          const void* const* src, cudaMemcpyKind kind, cudaStream_t st)
{
    const int64_t row = p.N * p.d * p.e;
    for (int q = 0; q < p.W; ++q) {
        if (rows.cnt[q] == 0) continue;
        for (int64_t bb = 0; bb < p.b; ++bb) {
            const int64_t off = (bb * p.s[q] + rows.lo[q]) * row;
            cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t*>(dst[q]) + off,
                                            static_cast<const uint8_t*>(src[q]) + off,
                                            size_t(rows.cnt[q] * row), kind, st);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

// The same rows on every rank's head-side tensor (b, S, n_r, d): rows seq_off(q) + [lo_q, ...).
cudaError_t copy_head_rows(const Plan& p, const ChunkRows& rows, void* const* dst,
                           const void* const* src, cudaMemcpyKind kind, cudaStream_t st)
{
    for (int r = 0; r < p.W; ++r) {
        const int64_t row = p.n[r] * p.d * p.e;
        if (row == 0) continue;
        for (int64_t bb = 0; bb < p.b; ++bb)
            for (int q = 0; q < p.W; ++q) {
                if (rows.cnt[q] == 0) continue;
                const int64_t off = (bb * p.S + p.seq_off[q] + rows.lo[q]) * row;
                cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t*>(dst[r]) + off,
                                                static_cast<const uint8_t*>(src[r]) + off,
                                                size_t(rows.cnt[q] * row), kind, st);
                if (e != cudaSuccess) return e;
            }
    }
    return cudaSuccess;
}

// The host pipeline cuts the global sequence into ranges of `span` rows (about kPipeChunks of
// them, within the chunk cap): a range touches one or two sequence shards and is one contiguous
// span of every head-side tensor, so each chunk needs few, large copies. (Measured on a GB300:
// eight equal ranges beat 4, 6, 12, 16 and 32, and beat short first and last ranges around
// equal middle ones, which cost 5% more per call although they shorten the time one copy
// direction runs alone.)
struct PipeChunks {
    int64_t span = 0;
    int64_t count(const Plan& p) const { return (p.S + span - 1) / span; }
    void rows(const Plan& p, int64_t c, ChunkRows* out) const
    {
        const int64_t lo = c * span;
        global_chunk_rows(p, lo, lo + span < p.S ? lo + span : p.S, out);
    }
};

int pipe_chunks(const Plan& p, PipeChunks* pc)
{
    pc->span = global_chunk_span(p, kPipeChunks);
    return pc->span > 0 ? ULY_OK : ULY_ECHUNK;
}

// One call through the pipeline: copy_in(rows, stream) for each range on the input stream,
// kernel(rows, stream) on the caller's stream, copy_out(rows, stream) on the output stream.
template <class CopyIn, class Kernel, class CopyOut>
int run_host_pipe(const Plan& p, const PipeChunks& pc, HostPipe* hp, cudaStream_t st,
                  CopyIn copy_in, Kernel kernel, CopyOut copy_out)
{
    // copies in overwrite the caller's device inputs: after everything already queued on `st`
    cudaError_t e = cudaEventRecord(hp->entry, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->in, hp->entry, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    const int64_t C = pc.count(p);
    for (int64_t c = 0; c < C; ++c) {
        ChunkRows rows;
        pc.rows(p, c, &rows);
        if ((e = copy_in(rows, hp->in)) != cudaSuccess) return cuda_fail(e);
        cudaEvent_t in_done = hp->in_done[c % kPipeEvents];
        if ((e = cudaEventRecord(in_done, hp->in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(st, in_done, 0)) != cudaSuccess)
            return cuda_fail(e);
        const int rc = kernel(rows, st);
        if (rc) return rc;
        cudaEvent_t done = hp->chunk_done[c % kPipeEvents];
        if ((e = cudaEventRecord(done, st)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(hp->aux, done, 0)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = copy_out(rows, hp->aux)) != cudaSuccess) return cuda_fail(e);
    }
    e = cudaEventRecord(hp->copied_out, hp->aux);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hp->copied_out, 0);
    return e == cudaSuccess ? ULY_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

int ulysses_plan(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits, int64_t d,
                 int dtype, ulysses_plan_t* out)
{
    if (!out) return ULY_EINVAL;
    *out = nullptr;
    Plan p;
    const int rc = plan_init(&p, W, b, seq_splits, head_splits, d, dtype);
    if (rc) return rc;
    ulysses_plan_s* h = new (std::nothrow) ulysses_plan_s;
    if (!h) return ULY_ENOMEM;
    h->p = p;
    *out = h;
    return ULY_OK;
}

int ulysses_plan_destroy(ulysses_plan_t plan)
{
    delete plan;
    return ULY_OK;
}

int ulysses_plan_set_chunk_bytes(ulysses_plan_t plan, int64_t max_chunk_bytes)
{
    if (!plan || max_chunk_bytes < 1) return ULY_EINVAL;
    plan->p.chunk_cap = max_chunk_bytes;
    return ULY_OK;
}

int ulysses_plan_set_rope_pairs(ulysses_plan_t plan, int pairs)
{
    if (!plan || (pairs != ULY_ROPE_ADJACENT && pairs != ULY_ROPE_HALF)) return ULY_EINVAL;
    plan->p.rope_half = pairs == ULY_ROPE_HALF ? 1 : 0;
    return ULY_OK;
}

int ulysses_plan_set_fused_engine(ulysses_plan_t plan, int engine)
{
    if (!plan || (engine != ULY_ENGINE_AUTO && engine != ULY_ENGINE_TMA && engine != ULY_ENGINE_TENSOR))
        return ULY_EINVAL;
    plan->p.fused_engine = engine;
    return ULY_OK;
}

int ulysses_plan_fused_kernel(ulysses_plan_t plan, int* engine)
{
    if (!plan || !engine) return ULY_EINVAL;
    *engine = fused_uses_tensor(plan->p) ? ULY_ENGINE_TENSOR : ULY_ENGINE_TMA;
    return ULY_OK;
}

int ulysses_plan_fused_backward_kernel(ulysses_plan_t plan, int* engine)
{
    if (!plan || !engine) return ULY_EINVAL;
    *engine = fused_bwd_uses_group_major(plan->p) ? ULY_ENGINE_TENSOR : ULY_ENGINE_TMA;
    return ULY_OK;
}

int ulysses_plan_set_max_ctas(ulysses_plan_t plan, int64_t max_ctas)
{
    if (!plan || max_ctas < 0) return ULY_EINVAL;
    plan->p.max_ctas = max_ctas;
    return ULY_OK;
}

int ulysses_plan_bytes(ulysses_plan_t plan, int mode, int rank, int64_t* in_bytes, int64_t* out_bytes)
{
    if (!plan || (mode != 0 && mode != 1) || rank < 0 || rank >= plan->p.W) return ULY_EINVAL;
    const int64_t sq = seq_side_bytes(plan->p, rank), hd = head_side_bytes(plan->p, rank);
    if (in_bytes) *in_bytes = mode == 0 ? sq : hd;
    if (out_bytes) *out_bytes = mode == 0 ? hd : sq;
    return ULY_OK;
}

int ulysses_plan_auto_engine(ulysses_plan_t plan, int* engine)
{
    if (!plan || !engine) return ULY_EINVAL;
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc) return rc;
    *engine = relayout_tensor_preferred(plan->p, dev.sm_count) ? ULY_ENGINE_TENSOR : ULY_ENGINE_TMA;
    return ULY_OK;
}

int ulysses_plan_num_chunks(ulysses_plan_t plan, int mode, int64_t* n_chunks)
{
    if (!plan || !n_chunks || (mode != 0 && mode != 1)) return ULY_EINVAL;
    return num_chunks(plan->p, n_chunks);
}

int ulysses_plan_chunk_rows(ulysses_plan_t plan, int mode, int64_t chunk, int64_t* row_lo,
                            int64_t* row_count)
{
    if (!plan || !row_lo || !row_count || (mode != 0 && mode != 1)) return ULY_EINVAL;
    int64_t C = 0;
    const int rc = num_chunks(plan->p, &C);
    if (rc) return rc;
    if (chunk < 0 || chunk >= C) return ULY_EINVAL;
    ChunkRows rows;
    chunk_rows(plan->p, C, chunk, &rows);
    for (int q = 0; q < plan->p.W; ++q) {
        row_lo[q] = rows.lo[q];
        row_count[q] = rows.cnt[q];
    }
    return ULY_OK;
}

int ulysses_plan_rank_segments(ulysses_plan_t plan, int mode, int rank, ulysses_segment_t* segs)
{
    if (!plan || !segs || (mode != 0 && mode != 1)) return ULY_EINVAL;
    const Plan& p = plan->p;
    if (rank < 0 || rank >= p.W) return ULY_EINVAL;
    const int64_t de = p.d * p.e;
    for (int peer = 0; peer < p.W; ++peer) {
        // mode 0: rank q = `rank` sends head group r = peer of its sequence shard;
        // mode 1: rank r = `rank` sends sequence shard q = peer of its head group
        const int q = mode == 0 ? rank : peer;
        const int r = mode == 0 ? peer : rank;
        const int64_t seq_row = p.N * de;     // a row of rank q's (b, s_q, N, d)
        const int64_t head_row = p.n[r] * de; // a row of rank r's (b, S, n_r, d)
        const int64_t seq_at = p.head_off[r] * de, head_at = p.seq_off[q] * head_row;
        ulysses_segment_t& g = segs[peer];
        g.peer = peer;
        g.rows = p.s[q];
        g.row_bytes = p.n[r] * de;
        const int64_t sp[3] = {seq_at, seq_row, p.s[q] * seq_row};
        const int64_t hp[3] = {head_at, head_row, p.S * head_row};
        const int64_t* src = mode == 0 ? sp : hp;
        const int64_t* dst = mode == 0 ? hp : sp;
        g.src_offset = src[0];
        g.src_row_pitch = src[1];
        g.src_batch_pitch = src[2];
        g.dst_offset = dst[0];
        g.dst_row_pitch = dst[1];
        g.dst_batch_pitch = dst[2];
    }
    return ULY_OK;
}

int ulysses_a2a_4d(ulysses_plan_t plan, int mode, const void* const* in_ptrs, void* const* out_ptrs,
                   void* stream)
{
    if (!plan) return ULY_EINVAL;
    return relayout_impl(plan->p, mode, ULY_ENGINE_AUTO, in_ptrs, out_ptrs,
                         static_cast<cudaStream_t>(stream));
}

int ulysses_a2a_4d_engine(ulysses_plan_t plan, int mode, int engine, const void* const* in_ptrs,
                          void* const* out_ptrs, void* stream)
{
    if (!plan) return ULY_EINVAL;
    return relayout_impl(plan->p, mode, engine, in_ptrs, out_ptrs, static_cast<cudaStream_t>(stream));
}

int ulysses_a2a_4d_qk_fused(ulysses_plan_t plan, const void* const* q_in, const void* const* k_in,
                            void* const* q_out, void* const* k_out, const float* rms_w, float eps,
                            float rope_theta, void* stream)
{
    if (!plan) return ULY_EINVAL;
    return fused_device(plan->p, q_in, k_in, q_out, k_out, nullptr, rms_w, eps, rope_theta,
                        static_cast<cudaStream_t>(stream));
}

int ulysses_qk_fused_backward_workspace(ulysses_plan_t plan, size_t* bytes)
{
    if (!plan || !bytes) return ULY_EINVAL;
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    int64_t T = 0;
    int stages = 0, ctas_per_sm = 1;
    uint32_t stage_bytes = 0;
    return fused_bwd_setup(plan->p, dev, &T, &stages, &stage_bytes, &ctas_per_sm, bytes);
}

int ulysses_a2a_4d_qk_fused_backward(ulysses_plan_t plan, void* const* dq_out, void* const* dk_out,
                                     const void* const* q_in, const void* const* k_in,
                                     const void* const* dq_in, const void* const* dk_in,
                                     const float* rms_w, float* dw, float eps, float rope_theta,
                                     void* workspace, size_t workspace_bytes, void* stream)
{
    if (!plan) return ULY_EINVAL;
    return fused_bwd_device(plan->p, dq_out, dk_out, q_in, k_in, dq_in, dk_in, rms_w, dw, eps,
                            rope_theta, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int ulysses_a2a_4d_qkv_fused_backward(ulysses_plan_t plan, void* const* dqkv_out,
                                      const void* const* qkv_in, const void* const* dq_in,
                                      const void* const* dk_in, const void* const* dv_in,
                                      const float* rms_w, float* dw, float eps, float rope_theta,
                                      void* workspace, size_t workspace_bytes, void* stream)
{
    if (!plan || !qkv_in || !dqkv_out || !dq_in || !dk_in || !dv_in) return ULY_EINVAL;
    const Plan& p = plan->p;
    const void* grads[3 * kMaxW];
    for (int k = 0; k < p.W; ++k) {
        grads[k] = dq_in[k];
        grads[p.W + k] = dk_in[k];
        grads[2 * p.W + k] = dv_in[k];
    }
    return packed_bwd_device(p, dqkv_out, qkv_in, 3, 0, 1, 3 * p.N * p.d * p.e, grads, rms_w, dw,
                             eps, rope_theta, workspace, workspace_bytes,
                             static_cast<cudaStream_t>(stream));
}

int ulysses_a2a_4d_packed_fused_backward(ulysses_plan_t plan, int planes, int q_plane,
                                         int k_plane, int64_t token_pitch,
                                         void* const* dpacked_out, const void* const* packed_in,
                                         const void* const* grads, const float* rms_w, float* dw,
                                         float eps, float rope_theta, void* workspace,
                                         size_t workspace_bytes, void* stream)
{
    if (!plan) return ULY_EINVAL;
    return packed_bwd_device(plan->p, dpacked_out, packed_in, planes, q_plane, k_plane,
                             token_pitch, grads, rms_w, dw, eps, rope_theta, workspace,
                             workspace_bytes, static_cast<cudaStream_t>(stream));
}

int ulysses_a2a_4d_qk_fused_backward_static(ulysses_plan_t plan, void* const* dq_out,
                                            void* const* dk_out, const void* const* q_in,
                                            const void* const* k_in, const void* const* dq_in,
                                            const void* const* dk_in, const float* rms_w,
                                            float* dw, float eps, float rope_theta, void* stream)
{
    if (!plan) return ULY_EINVAL;
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    int64_t T = 0;
    int stages = 0, ctas_per_sm = 1;
    uint32_t stage_bytes = 0;
    size_t need = 0;
    if ((rc = fused_bwd_setup(plan->p, dev, &T, &stages, &stage_bytes, &ctas_per_sm, &need)))
        return rc;
    if (need > ULYSSES_STATIC_SCRATCH_BYTES) return ULY_ESCRATCH;
    void* scratch = nullptr;
    if ((rc = static_scratch(dev.device, &scratch))) return rc;
    return fused_bwd_device(plan->p, dq_out, dk_out, q_in, k_in, dq_in, dk_in, rms_w, dw, eps,
                            rope_theta, scratch, ULYSSES_STATIC_SCRATCH_BYTES,
                            static_cast<cudaStream_t>(stream));
}

int ulysses_a2a_4d_qkv_fused(ulysses_plan_t plan, const void* const* qkv_in, void* const* q_out,
                             void* const* k_out, void* const* v_out, const float* rms_w, float eps,
                             float rope_theta, void* stream)
{
    if (!plan || !qkv_in || !q_out || !k_out || !v_out) return ULY_EINVAL;
    const Plan& p = plan->p;
    void* outs[3 * kMaxW];
    for (int k = 0; k < p.W; ++k) {
        outs[k] = q_out[k];
        outs[p.W + k] = k_out[k];
        outs[2 * p.W + k] = v_out[k];
    }
    const PackedIn pk{qkv_in, 3, 0, 1, 3 * p.N * p.d * p.e, outs};
    return fused_device(p, nullptr, nullptr, nullptr, nullptr, &pk, rms_w, eps, rope_theta,
                        static_cast<cudaStream_t>(stream));
}

int ulysses_a2a_4d_packed_fused(ulysses_plan_t plan, int planes, int q_plane, int k_plane,
                                int64_t token_pitch, const void* const* packed_in,
                                void* const* outs, const float* rms_w, float eps, float rope_theta,
                                void* stream)
{
    if (!plan || !packed_in || !outs) return ULY_EINVAL;
    const PackedIn pk{packed_in, planes, q_plane, k_plane, token_pitch, outs};
    return fused_device(plan->p, nullptr, nullptr, nullptr, nullptr, &pk, rms_w, eps, rope_theta,
                        static_cast<cudaStream_t>(stream));
}

int ulysses_a2a_4d_host(ulysses_plan_t plan, int mode, const void* const* host_in,
                        void* const* host_out, void* const* dev_in, void* const* dev_out, void* stream)
{
    if (!plan || !host_in || !host_out || !dev_in || !dev_out) return ULY_EINVAL;
    const Plan& p = plan->p;
    if (mode != 0 && mode != 1) return ULY_EINVAL;
    int64_t in_b[kMaxW], out_b[kMaxW];
    side_bytes(p, mode, in_b, out_b);
    for (int k = 0; k < p.W; ++k) {
        if ((in_b[k] && !host_in[k]) || (out_b[k] && !host_out[k])) return ULY_EINVAL;
    }
    // validate the device side before queuing any copy
    int rc = check_ptrs(const_cast<const void* const*>(dev_in), in_b, p.W);
    if (rc) return rc;
    rc = check_ptrs(const_cast<const void* const*>(dev_out), out_b, p.W);
    if (rc) return rc;
    rc = check_overlap(const_cast<const void* const*>(dev_in), in_b, p.W,
                       const_cast<const void* const*>(dev_out), out_b, p.W);
    if (rc) return rc;
    PipeChunks pc;
    if ((rc = pipe_chunks(p, &pc))) return rc;
    DeviceInfo dev;
    if ((rc = current_device(&dev))) return rc;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe* hp = nullptr;
    if ((rc = host_pipe(dev.device, &hp))) return rc;
    const void* const* din = const_cast<const void* const*>(dev_in);
    const void* const* dout = const_cast<const void* const*>(dev_out);
    return run_host_pipe(
        p, pc, hp, static_cast<cudaStream_t>(stream),
        [&](const ChunkRows& rows, cudaStream_t s) {
            return mode == 0 ? copy_seq_rows(p, rows, dev_in, host_in, cudaMemcpyHostToDevice, s)
                             : copy_head_rows(p, rows, dev_in, host_in, cudaMemcpyHostToDevice, s);
        },
        [&](const ChunkRows& rows, cudaStream_t s) {
            return relayout_rows(p, mode, ULY_ENGINE_AUTO, din, dev_out, rows, s, dev);
        },
        [&](const ChunkRows& rows, cudaStream_t s) {
            return mode == 0 ? copy_head_rows(p, rows, host_out, dout, cudaMemcpyDeviceToHost, s)
                             : copy_seq_rows(p, rows, host_out, dout, cudaMemcpyDeviceToHost, s);
        });
}

int ulysses_a2a_4d_qk_fused_host(ulysses_plan_t plan, const void* const* q_host_in,
                                 const void* const* k_host_in, void* const* q_host_out,
                                 void* const* k_host_out, void* const* q_in, void* const* k_in,
                                 void* const* q_out, void* const* k_out, const float* rms_w,
                                 float eps, float rope_theta, void* stream)
{
    if (!plan || !q_host_in || !k_host_in || !q_host_out || !k_host_out || !q_in || !k_in)
        return ULY_EINVAL;
    const Plan& p = plan->p;
    int64_t in_b[kMaxW], out_b[kMaxW];
    side_bytes(p, 0, in_b, out_b);
    for (int k = 0; k < p.W; ++k) {
        if ((in_b[k] && (!q_host_in[k] || !k_host_in[k])) ||
            (out_b[k] && (!q_host_out[k] || !k_host_out[k])))
            return ULY_EINVAL;
    }
    FusedArgs a;
    int64_t T = 0;
    int rc = fused_prepare(p, const_cast<const void* const*>(q_in), const_cast<const void* const*>(k_in),
                           q_out, k_out, nullptr, rms_w, eps, rope_theta, &a, &T);
    if (rc) return rc;
    PipeChunks pc;
    if ((rc = pipe_chunks(p, &pc))) return rc;
    DeviceInfo dev;
    if ((rc = current_device(&dev))) return rc;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe* hp = nullptr;
    if ((rc = host_pipe(dev.device, &hp))) return rc;
    const void* const* qo = const_cast<const void* const*>(q_out);
    const void* const* ko = const_cast<const void* const*>(k_out);
    return run_host_pipe(
        p, pc, hp, static_cast<cudaStream_t>(stream),
        [&](const ChunkRows& rows, cudaStream_t s) {
            cudaError_t e = copy_seq_rows(p, rows, q_in, q_host_in, cudaMemcpyHostToDevice, s);
            return e == cudaSuccess ? copy_seq_rows(p, rows, k_in, k_host_in, cudaMemcpyHostToDevice, s)
                                    : e;
        },
        [&](const ChunkRows& rows, cudaStream_t s) { return fused_rows(p, &a, T, rows, s, dev); },
        [&](const ChunkRows& rows, cudaStream_t s) {
            cudaError_t e = copy_head_rows(p, rows, q_host_out, qo, cudaMemcpyDeviceToHost, s);
            return e == cudaSuccess ? copy_head_rows(p, rows, k_host_out, ko, cudaMemcpyDeviceToHost, s)
                                    : e;
        });
}

int ulysses_device_status(unsigned* status)
{
    if (!status) return ULY_EINVAL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned a = 0, b = 0, c = 0, t = 0;
    if ((e = relayout_status(&a, true)) != cudaSuccess) return cuda_fail(e);
    if ((e = fused_status(&b, true)) != cudaSuccess) return cuda_fail(e);
    if ((e = fused_bwd_status(&c, true)) != cudaSuccess) return cuda_fail(e);
    if ((e = fused_tensor_status(&t, true)) != cudaSuccess) return cuda_fail(e);
    *status = a | b | c | t;
    return *status ? ULY_EDEVICE : ULY_OK;
}

int ulysses_selftest_wait_timeout(unsigned limit_us, void* stream)
{
    if (limit_us < 1 || limit_us > 1000000u) return ULY_EINVAL;
    cudaError_t e = selftest_timeout_launch(uint64_t(limit_us) * 1000u, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ULY_OK : cuda_fail(e);
}

int ulysses_last_cuda_error(void) { return t_last_cuda_error; }

const char* ulysses_strerror(int status)
{
    switch (status) {
        case ULY_OK: return "ok";
        case ULY_EINVAL: return "invalid argument";
        case ULY_EALIGN: return "misaligned pointer or d * elem_size not a multiple of 16";
        case ULY_EOVERLAP: return "output range overlaps an input or another output";
        case ULY_ECHUNK: return "chunk cap smaller than one sequence row";
        case ULY_ECUDA: return "CUDA runtime error (see ulysses_last_cuda_error)";
        case ULY_ENOMEM: return "out of host memory";
        case ULY_EDEVICE: return "a kernel wait timed out (device status word set)";
        case ULY_ESCRATCH: return "needs more scratch than the library's static array holds";
        default: return "unknown status";
    }
}

int ulysses_version(void) { return 100; }

}  // extern "C"
