// Segments of the stream-K split's lines (shared by the shared-prefix decode
// kernel and its tensor-core prefix line): the stretch of one row (a sequence's
// suffix or a group's shared blocks) that a CTA's range of units covers.
#pragma once

namespace pa {

// The segment of a line that starts at unit u (u inside the line, u < end).
struct Segment {
  int row;            // sequence (suffix line) or group (prefix line)
  int kvg;            // KV head group
  int b0;             // first block, counted from the row's first (shared) block
  int nblk;           // blocks in the segment
  bool whole;         // the segment is its row's whole range
  bool first;         // the segment starts the CTA's range (cut slot 0, else 1)
  bool row_end;       // the segment reaches its row's last block
};

// The segment of a KV head group's line that starts at unit u (u < u_end).
// Unit counts fit in 32 bits: the host admits a call only if (sequences +
// groups) x max_blocks_per_seq x num_kv_heads < 2^31.
__device__ __forceinline__ Segment segment_at(int u, int u_begin, int u_end, const int* base,
                                              int nrows, const int* first_blk) {
  // the row r with base[r] <= u < base[r + 1] (rows of no units skipped)
  int lo = 0, hi = nrows - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (base[mid + 1] > u) hi = mid; else lo = mid + 1;
  }
  Segment s;
  s.row = lo;
  s.kvg = 0;  // set by the caller: a CTA's line belongs to one KV head group
  const int row_start = base[lo];
  const int row_stop = base[lo + 1];
  const int seg_end = min(row_stop, u_end);
  s.b0 = (first_blk ? first_blk[lo] : 0) + (u - row_start);
  s.nblk = seg_end - u;
  s.whole = (u == row_start) && (seg_end == row_stop);
  s.first = (u == u_begin);
  s.row_end = (seg_end == row_stop);
  return s;
}

}  // namespace pa
