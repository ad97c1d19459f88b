// tensor_map.h -- tiled tensor maps for the kernels that move one head group's runs of a block of
// sequence rows with a single cp.async.bulk.tensor copy.
#pragma once

#include <cuda.h>  // CUtensorMap and the encoder's types (the encoder is fetched at run time)

#include <cstdint>

namespace uly {

// A 3-D map over one (shard, head group) segment of a (b, s, N, d) tensor: eight-byte elements
// x rows x batch. `base` is the segment's first byte (16-byte aligned), `run` its bytes per row (a
// multiple of 16, at most 2,048: the box's inner extent is 256 elements at most), `rows` and `b`
// its extents, `row_stride` and `batch_stride` the byte strides of a row and a batch index
// (multiples of 16), `box_rows` (1..256) the rows one copy moves. Every box starts at x = 0.
// Returns false when the driver provides no encoder or rejects the map.
bool encode_run_map(CUtensorMap* map, const void* base, int64_t run, int64_t rows, int64_t b,
                    int64_t row_stride, int64_t batch_stride, int64_t box_rows);

// A 4-D map over the rows of one shard of a (b, s, N, d) tensor whose W head groups all have the
// same run: eight-byte elements x rows x head group x batch, with strides row_stride (N d e),
// run (one group to the next) and batch_stride. A box (run / 8, box_rows, W, 1) lands in shared
// memory group-major, [group][row][run]: the rows of each destination rank back to back, as its
// head-side tensor holds them.
bool encode_group_map(CUtensorMap* map, const void* base, int64_t run, int64_t rows, int64_t W,
                      int64_t b, int64_t row_stride, int64_t batch_stride, int64_t box_rows);

}  // namespace uly
