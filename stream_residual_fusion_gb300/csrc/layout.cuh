// layout.cuh -- geometry of the fused step's pipeline stages, shared by the fused kernel and the
// weight-packing kernel (the packed weights are stored as the exact shared-memory image that the
// fused kernel's tensor-core operand tiles need, so one contiguous bulk copy brings a stage's
// weights).
#pragma once
#include <cstdint>

namespace mhc {

constexpr int STEP_TT = 128;     // tokens per tile (the MMA's M)
constexpr int STEP_DC = 32;      // columns of d per pipeline stage
constexpr int STEP_ROW_BYTES = STEP_DC * 2;              // one bf16 tile row: 64 bytes
constexpr int STEP_CHUNKS = STEP_ROW_BYTES / 16;         // 16-byte chunks per tile row
constexpr int STEP_WROWS = 72;   // 3 bf16 planes x 24 mix rows
constexpr int STEP_MMA_N = 80;   // the MMA's N: weight rows 72..79 are zero
// one column block of the packed weights: 4 streams x [80 rows x DC columns]
constexpr int STEP_WSTREAM_BYTES = STEP_MMA_N * STEP_ROW_BYTES;
constexpr int STEP_WBLOCK_BYTES = 4 * STEP_WSTREAM_BYTES;

// Byte offset of 16-byte chunk `chunk` of row `row` in a K-major operand tile with STEP_DC
// columns, stored with the hardware swizzle whose width is the row size (32, 64 or 128 bytes):
// chunk c of row r sits at chunk c ^ ((r * row_bytes / 128) mod chunks_per_row).
__host__ __device__ constexpr uint32_t tile_chunk_offset(int row, int chunk) {
  return static_cast<uint32_t>(row * STEP_ROW_BYTES +
                               ((chunk ^ ((row * STEP_ROW_BYTES >> 7) & (STEP_CHUNKS - 1))) << 4));
}

// Packed weight row of plane pl (0 hi, 1 mid, 2 lo) of mix row r: each half of the 24 mix rows
// keeps its three planes together, so a thread folding 12 mix numbers reads 36 adjacent columns
// of the accumulator.
__host__ __device__ constexpr int packed_row(int r, int pl) { return 36 * (r / 12) + 12 * pl + r % 12; }

}  // namespace mhc
