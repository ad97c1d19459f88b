// plan.h -- host plan of the Ulysses 4D relayout and the by-value argument blocks its kernels
// receive. Shared by plan.cpp (host only, no CUDA calls) and the .cu files.
#pragma once
#include <cuda.h>  // CUtensorMap

#include <cstdint>

namespace uly {

constexpr int kMaxW = 8;
constexpr int kMaxSeg = kMaxW * kMaxW;
constexpr int kMaxFusedD = 256;

struct Plan {
    int W;
    int dtype;
    int64_t b, d, e;  // batch, head dim, element bytes
    int64_t S, N;     // global sequence length, global head count
    int64_t s[kMaxW], n[kMaxW];
    int64_t seq_off[kMaxW + 1], head_off[kMaxW + 1];
    int64_t chunk_cap;  // max bytes one rank reads or writes per launch
    int64_t max_ctas;   // cap on the CTAs of any launch (0: none)
    int rope_half;      // the fused calls' RoPE pairs: (j, j + d/2) when set, else (2j, 2j + 1)
    int fused_engine;   // the fused forward's kernel: ULY_ENGINE_AUTO, _TMA (token units), _TENSOR
};

// Rows of each sequence shard covered by one launch.
struct ChunkRows {
    int64_t lo[kMaxW];
    int64_t cnt[kMaxW];
};

int64_t elem_size_of(int dtype);  // 0 for an unknown dtype
int plan_init(Plan* p, int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
              int64_t d, int dtype);  // ULY_* status
int64_t seq_side_bytes(const Plan& p, int q);   // rank q's (b, s_q, N, d) tensor
int64_t head_side_bytes(const Plan& p, int r);  // rank r's (b, S, n_r, d) tensor
int num_chunks(const Plan& p, int64_t* n_chunks);  // ULY_OK or ULY_ECHUNK
void chunk_rows(const Plan& p, int64_t n_chunks, int64_t chunk, ChunkRows* out);
// Rows of each shard inside the global sequence range [lo, hi) (the shards tile [0, S) in rank
// order): a range touches few shards and is contiguous on every head-side tensor.
void global_chunk_rows(const Plan& p, int64_t lo, int64_t hi, ChunkRows* out);
// Global rows per range so that about target_chunks ranges cover S and no rank reads or writes
// more than the chunk cap in one launch; 0 when one global row already exceeds the cap.
int64_t global_chunk_span(const Plan& p, int64_t target_chunks);

// ---- relayout kernels' argument block (passed by value, lives in the parameter bank) ----------
// A work unit is a block of up to rows_per_unit[r] consecutive rows of one segment (q, r) and one
// batch index, or, when one row's run (n_r * d * e bytes) exceeds unit_bytes, a unit_bytes-wide
// piece of a single row. "Seq side" is rank q's (b, s_q, N, d) tensor (mode 0 reads it, mode 1
// writes it); "head side" is rank r's (b, S, n_r, d) tensor.
struct RelayoutArgs {
    uint8_t* seq_ptr[kMaxW];
    uint8_t* head_ptr[kMaxW];
    int64_t s[kMaxW], seq_off[kMaxW], n[kMaxW], head_off[kMaxW];
    int64_t row_lo[kMaxW], rows[kMaxW];          // this launch's rows of shard q
    int64_t rows_per_unit[kMaxW], pieces[kMaxW];  // per destination head group r
    int64_t unit_begin[kMaxSeg + 1];              // prefix of unit counts over g = q * W + r
    int64_t S, N, b, d_bytes;
    int64_t total_units;
    int32_t W, unit_bytes;
};

// Fills the unit tables of `a` for one launch (pointers are set by the caller).
void build_relayout_units(const Plan& p, const ChunkRows& rows, int64_t unit_bytes, RelayoutArgs* a);

// ---- row-tile relayout argument block ---------------------------------------------------------
// A work unit is up to tile_rows consecutive rows (tokens) of one sequence shard q and one batch
// index, with all N heads: on the sequence side one contiguous span of tile_rows * N * d * e bytes,
// on the head side W contiguous spans (one per rank r, tile_rows * n_r * d * e bytes each). Used
// when a whole row fits a shared-memory stage.
struct RowTileArgs {
    uint8_t* seq_ptr[kMaxW];
    uint8_t* head_ptr[kMaxW];
    int64_t s[kMaxW], seq_off[kMaxW], n[kMaxW], head_off[kMaxW];
    int64_t row_lo[kMaxW], rows[kMaxW];
    int64_t unit_begin[kMaxW + 1];  // prefix of unit counts over q
    int64_t S, N, b, d_bytes;
    int64_t tile_rows, total_units;
    int32_t W;
    int32_t stage_bytes;  // bytes between consecutive stages in shared memory
};

// Shape of the row-tile kernel's pipeline for one plan and mode, chosen on the host from the
// geometry (relayout_row_ring): loads in flight ahead of the unit being stored, CTAs per SM and
// the bytes of one stage (the ring always has kRowStages stages).
constexpr int kRowStages = 4;
struct RowRing {
    int lookahead;
    int ctas_per_sm;
    int stage_bytes;
};

void build_row_tiles(const Plan& p, const ChunkRows& rows, int64_t tile_rows, RowTileArgs* a);

// ---- fused QK kernel's argument block ---------------------------------------------------------
// Work is cut into blocks of `block_tokens` consecutive source rows (tokens) of one shard q and one
// batch index, and each block into `units_per_block` work units:
//  * separate q and k inputs: one unit per block (block_tokens = tokens_per_unit), all N heads of
//    q and of k for those tokens;
//  * `interleaved` (packed_in[q]: rank q's b * s_q tokens, tok_pitch bytes apart, each holding
//    `planes` planes of N * d elements, plane c at byte c * N * d * e of the token): blocks of
//    2 * tokens_per_unit tokens with `planes` units each: the q and k rows (planes q_plane and
//    k_plane) of its first tokens_per_unit tokens, those of the next tokens_per_unit, and one unit
//    per other plane (plain_plane[0 .. planes - 3], in order) with that plane's rows of all the
//    block's tokens, which plane_out receives unchanged. Each unit fills the same stage size.
//    Units 0 .. 2B-1 (B blocks) are the q,k units (two per block, in block order), then B units of
//    each plain plane in turn.
// unit_begin counts blocks; total_units counts units.
constexpr int kMaxPlanes = 8;
struct FusedArgs {
    const uint8_t* q_in[kMaxW];
    const uint8_t* k_in[kMaxW];
    const uint8_t* packed_in[kMaxW];
    uint8_t* q_out[kMaxW];
    uint8_t* k_out[kMaxW];
    uint8_t* plane_out[kMaxPlanes][kMaxW];  // the plain planes' outputs (packed calls)
    int32_t interleaved;
    int32_t planes, q_plane, k_plane;   // packed calls
    int32_t plain_plane[kMaxPlanes];    // the planes other than q and k, in order
    int64_t tok_pitch;                  // packed calls: bytes between consecutive tokens
    int32_t elem_f16;   // elements are fp16 (else bf16)
    int32_t rope_half;  // RoPE pairs (j, j + d/2) (else (2j, 2j + 1))
    const float* rms_w;  // [2][d]
    int64_t s[kMaxW], seq_off[kMaxW], n[kMaxW], head_off[kMaxW];
    int64_t row_lo[kMaxW], rows[kMaxW];
    int64_t unit_begin[kMaxW + 1];
    int64_t blocks[kMaxW];  // token blocks per batch index of shard q
    int64_t S, N, b;
    int64_t total_units;
    int32_t W, d, tokens_per_unit, stages;
    int32_t block_tokens, units_per_block;
    int32_t ctas_per_sm;  // resident CTAs per SM the shared-memory footprint allows
    uint32_t stage_bytes;
    float eps;
    // theta^(-2j/d) / (2 pi) as an unevaluated sum hi + lo of two floats, j < d/2.
    float turn_hi[kMaxFusedD / 2];
    float turn_lo[kMaxFusedD / 2];
};
static_assert(sizeof(FusedArgs) <= 4096, "kernel parameter block");

void build_fused_units(const Plan& p, const ChunkRows& rows, int64_t tokens_per_unit,
                       int64_t block_tokens, int units_per_block, FusedArgs* a);

// ---- fused QK backward's argument block -------------------------------------------------------
// A token block is tokens_per_unit consecutive rows (tokens) of one shard q and one batch index;
// it makes one work unit per tensor (for q, k: unit u is tensor u mod 2 of block u div 2; for a
// packed call with C planes: unit u is tensor u div B of block u mod B, B blocks, tensors 0 and 1
// being the q and k planes and tensors 2 .. C-1 the other planes). A unit reads the tensor's
// forward input for those tokens (all N heads: one contiguous span on the sequence side) and the
// gradient of its output (W runs, rank r's n_r heads of those tokens, contiguous on rank r's head
// side), and writes the gradient of the input (one span on the sequence side).
// For a packed call the forward input and the gradient are rank q's packed tokens: x_in / dx_out
// point at a rank's plane and consecutive tokens are tok_stride bytes (the token pitch) apart;
// units of tensors 2 and up only gather their gradient (mode 1).
struct FusedBwdArgs {
    const uint8_t* x_in[2][kMaxW];           // forward inputs q, k: rank q's (b, s_q, N, d)
    const uint8_t* g_in[kMaxPlanes][kMaxW];  // gradients of the forward outputs: (b, S, n_r, d)
    uint8_t* dx_out[kMaxPlanes][kMaxW];      // gradients of the forward inputs: (b, s_q, N, d)
    int32_t tensors;                // 2 (q, k) or the packed call's planes
    int32_t tok_stride;             // bytes between consecutive tokens of x_in / dx_out
    const float* rms_w;             // [2][d]
    float* dw_part;                 // [grid][2][d]: one slot per CTA, fully written by it
    int32_t elem_f16;               // elements are fp16 (else bf16)
    int32_t rope_half;              // RoPE pairs (j, j + d/2) (else (2j, 2j + 1))
    int64_t s[kMaxW], seq_off[kMaxW], n[kMaxW], head_off[kMaxW + 1];
    int64_t row_lo[kMaxW], rows[kMaxW];
    int64_t block_begin[kMaxW + 1];  // prefix of token-block counts over q
    int64_t blocks[kMaxW];           // token blocks per batch index of shard q
    int64_t S, N, b;
    int64_t total_units;  // `tensors` per token block
    int32_t W, d, tokens_per_unit, stages;
    int32_t ctas_per_sm;
    uint32_t stage_bytes;  // forward input then output gradient of tokens_per_unit tokens
    float eps;
    float turn_hi[kMaxFusedD / 2];
    float turn_lo[kMaxFusedD / 2];
    // Row blocks (equal head groups): a unit's forward input arrives with one 4-D tensor-map copy
    // that lands it grouped by head group, [group][row][run], and its gradient with one copy per
    // rank in the same order (see encode_group_map).
    int32_t group_major;
    int32_t n_eq;     // heads per rank (all ranks equal) when group_major
    uint32_t run;     // n_eq * d * elem_size
    CUtensorMap xmap[2][kMaxW];  // q, k: per shard, this launch's rows
    CUtensorMap dmap[kMaxPlanes - 2][kMaxW];  // packed calls: the other planes' gradient outputs
};
static_assert(sizeof(FusedBwdArgs) <= 32764, "kernel parameter block");

void build_fused_bwd_units(const Plan& p, const ChunkRows& rows, int64_t tokens_per_unit,
                           FusedBwdArgs* a);
void rope_turns(int64_t d, double theta, float* turn_hi, float* turn_lo);

}  // namespace uly

struct ulysses_plan_s {
    uly::Plan p;
};
