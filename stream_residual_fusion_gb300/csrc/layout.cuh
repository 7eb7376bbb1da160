// layout.cuh -- geometry of the fused step's pipeline, shared by the fused kernel and the
// weight-packing kernel (the packed weights are stored as the exact shared-memory image that the
// fused kernel's tensor-core operand tiles need, so one contiguous bulk copy brings a block of
// weights).
#pragma once
#include <cstdint>

namespace mhc {

// A pipeline slot is STEP_TT token rows of STEP_DC columns of X_0..X_3 and F: 40 KB, so four
// slots fit in shared memory. (Slots of 64 tokens x 64 columns, the same 40 KB with 128-byte
// rows that DRAM serves better, measured slower at d = 5120: each slot then takes 16 MMAs and a
// fold, every weight block serves half as many tokens, and each group walks twice the tiles.)
constexpr int STEP_TT = 128;     // token rows per tile (the MMA's M)
constexpr int STEP_DC = 32;
constexpr int STEP_ROW_BYTES = STEP_DC * 2;
constexpr int STEP_CHUNKS = STEP_ROW_BYTES / 16;         // 16-byte chunks per row

// Packed weights: blocks of STEP_WDC columns of every stream, each the B operand of one half
// of a slot's MMAs.
constexpr int STEP_WDC = 32;
constexpr int STEP_WROW_BYTES = STEP_WDC * 2;            // 64 bytes
constexpr int STEP_WCHUNKS = STEP_WROW_BYTES / 16;
constexpr int STEP_WROWS = 72;   // 3 bf16 planes x 24 mix rows
constexpr int STEP_MMA_N = 80;   // the MMA's N: weight rows 72..79 are zero
// one column block of the packed weights: 4 streams x [80 rows x STEP_WDC columns]
constexpr int STEP_WSTREAM_BYTES = STEP_MMA_N * STEP_WROW_BYTES;
constexpr int STEP_WBLOCK_BYTES = 4 * STEP_WSTREAM_BYTES;

// Byte offset of 16-byte chunk `chunk` of row `row` in a K-major operand tile with `row_bytes`
// per row (32, 64 or 128), stored with the hardware swizzle of that width: chunk c of row r sits
// at chunk c ^ ((r * row_bytes / 128) mod chunks_per_row).
__host__ __device__ constexpr uint32_t swizzled_chunk_offset(int row, int chunk, int row_bytes) {
  return static_cast<uint32_t>(row * row_bytes +
                               ((chunk ^ ((row * row_bytes >> 7) & (row_bytes / 16 - 1))) << 4));
}
// ... of an X/F tile (STEP_ROW_BYTES-byte rows) and of a packed weight tile (64-byte rows)
__host__ __device__ constexpr uint32_t tile_chunk_offset(int row, int chunk) {
  return swizzled_chunk_offset(row, chunk, STEP_ROW_BYTES);
}
__host__ __device__ constexpr uint32_t wtile_chunk_offset(int row, int chunk) {
  return swizzled_chunk_offset(row, chunk, STEP_WROW_BYTES);
}

// Packed weight row of plane pl (0 hi, 1 mid, 2 lo) of mix row r: each half of the 24 mix rows
// keeps its three planes together, so a thread folding 12 mix numbers reads 36 adjacent columns
// of the accumulator.
__host__ __device__ constexpr int packed_row(int r, int pl) { return 36 * (r / 12) + 12 * pl + r % 12; }

}  // namespace mhc
