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

// Operand fragments: numerals built the same way (low digits first).
int mpg_frag_a_coords(int lane, int i, int* row, int* col) {
  if (lane < 0 || lane > 31 || i < 0 || i > 7 || !row || !col) return -1;
  const int off = (i & 1) * 1 + (lane & 3) * 2 + (i >> 2) * 8 + (lane >> 2) * 16 + ((i >> 1) & 1) * 128;
  *row = off / 16;  // A is 16 columns wide, row-major
  *col = off % 16;
  return 0;
}

int mpg_frag_a_decode(int row, int col, int* lane, int* i) {
  if (row < 0 || row > 15 || col < 0 || col > 15 || !lane || !i) return -1;
  const int off = row * 16 + col;
  const int d0 = off % 2, tig = (off / 2) % 4, d2 = (off / 8) % 2, group = (off / 16) % 8, d4 = off / 128;
  *lane = group * 4 + tig;
  *i = d2 * 4 + d4 * 2 + d0;
  return 0;
}

int mpg_frag_b_coords(int lane, int i, int* k, int* n) {
  if (lane < 0 || lane > 31 || i < 0 || i > 3 || !k || !n) return -1;
  const int off = (i & 1) * 1 + (lane & 3) * 2 + (i >> 1) * 8 + (lane >> 2) * 16;
  *n = off / 16;    // B is 16 rows (k) tall, column-major
  *k = off % 16;
  return 0;
}

int mpg_frag_b_decode(int k, int n, int* lane, int* i) {
  if (k < 0 || k > 15 || n < 0 || n > 7 || !lane || !i) return -1;
  const int off = n * 16 + k;
  const int d0 = off % 2, tig = (off / 2) % 4, d2 = (off / 8) % 2, group = off / 16;
  *lane = group * 4 + tig;
  *i = d2 * 2 + d0;
  return 0;
}

// tcgen05 accumulator: with M = 128 (cta_group::1) row i of D is TMEM lane
// i of the CTA; with M = 256 (cta_group::2) rows 0-127 sit in the lanes of
// CTA rank 0 and rows 128-255 in those of rank 1.  Column j of D is TMEM
// column j (from the accumulator's base).  A warp reaches the lane quarter
// warp % 4 only; tcgen05.ld.32x32b gives lane t of the warp the value of TMEM
// lane 32*(warp % 4) + t, register r of column col_base + r.
namespace {
bool tmem_shape_ok(int m_shape) { return m_shape == 128 || m_shape == 256; }
}  // namespace

int mpg_tmem_acc_coords(int m_shape, int cta_rank, int warp, int lane, int reg, int col_base, int* row, int* col) {
  if (!tmem_shape_ok(m_shape) || cta_rank < 0 || cta_rank >= m_shape / 128 || warp < 0 || lane < 0 || lane > 31 ||
      reg < 0 || col_base < 0 || reg >= 512 || col_base >= 512 || col_base + reg >= 512 || !row || !col)
    return -1;
  *row = 128 * cta_rank + 32 * (warp % 4) + lane;
  *col = col_base + reg;
  return 0;
}

int mpg_tmem_acc_decode(int m_shape, int row, int col, int load_cols, int* cta_rank, int* warp, int* lane, int* reg,
                        int* col_base) {
  if (!tmem_shape_ok(m_shape) || row < 0 || row >= m_shape || col < 0 || col >= 512 || load_cols < 1 ||
      load_cols > 128 || (load_cols & (load_cols - 1)) != 0 || !cta_rank || !warp || !lane || !reg || !col_base)
    return -1;
  const int within = row % 128;   // the TMEM lane in the CTA that holds the row
  *cta_rank = row / 128;
  *warp = within / 32;            // the lowest warp index of that lane quarter
  *lane = within % 32;
  *col_base = col - col % load_cols;
  *reg = col % load_cols;
  return 0;
}

}  // extern "C"
