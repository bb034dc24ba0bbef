// Host decode of accumulator fragments ("feat(cuda-device): derive the
// m16n8k16 accumulator fragment layout", sections "The layout is a
// mixed-radix numeral" and "API").
//
// The row-major offset of value j of lane `lane` in the 16x8 tile is a
// mixed-radix numeral with digits (low to high) j&1 (range 2), lane%4 (4),
// lane/4 (8), j>>1 (2) and place values 1, 2, 8, 64.  Every function here
// works from that numeral: coordinates are the offset split into row and
// column, and the inverse reads the digits back out.
#include <cstdint>

#include "mpgemm.h"

namespace {

bool in_range(int lane, int j) { return lane >= 0 && lane < 32 && j >= 0 && j < 4; }

int numeral(int lane, int j) { return (j & 1) * 1 + (lane & 3) * 2 + (lane >> 2) * 8 + (j >> 1) * 64; }

}  // namespace

extern "C" {

int mpg_acc_offset(int lane, int j) { return in_range(lane, j) ? numeral(lane, j) : -1; }

int mpg_acc_coords(int lane, int j, int* row, int* col) {
  if (!in_range(lane, j) || !row || !col) return -1;
  const int off = numeral(lane, j);
  *row = off / 8;  // the tile is 8 columns wide
  *col = off % 8;
  return 0;
}

int mpg_acc_decode(int offset, int* lane, int* j) {
  if (offset < 0 || offset >= 128 || !lane || !j) return -1;
  const int d0 = offset % 2;          // j & 1
  const int tig = (offset / 2) % 4;   // lane % 4
  const int group = (offset / 8) % 8; // lane / 4
  const int d3 = offset / 64;         // j >> 1
  *lane = group * 4 + tig;
  *j = d3 * 2 + d0;
  return 0;
}

int64_t mpg_acc_matrix_offset(int lane, int j, int64_t tile_row, int64_t tile_col, int64_t row_stride,
                              int64_t limit) {
  if (!in_range(lane, j) || tile_row < 0 || tile_col < 0 || row_stride <= 0 || limit < 0) return -1;
  const int off = numeral(lane, j);
  const int64_t r = off / 8, c = off % 8;
  int64_t row, col, base, total;
  if (__builtin_add_overflow(tile_row, r, &row)) return -1;
  if (__builtin_add_overflow(tile_col, c, &col)) return -1;
  if (col >= row_stride) return -1;  // the column would spill into the next row
  if (__builtin_mul_overflow(row, row_stride, &base)) return -1;
  if (__builtin_add_overflow(base, col, &total)) return -1;
  if (total >= limit) return -1;
  return total;
}

int mpg_tmem_acc_coords(int warp, int lane, int reg, int col_base, int* row, int* col) {
  if (warp < 0 || lane < 0 || lane > 31 || reg < 0 || col_base < 0 || col_base + reg >= 512 || !row || !col)
    return -1;
  *row = 32 * (warp % 4) + lane;
  *col = col_base + reg;
  return 0;
}

}  // extern "C"
