// lsc_chunk.h -- what the two kernels of the chunked gated delta rule share:
// the chunk size, the per-(chunk, v head) workspace record that the
// preparation kernel writes and the state kernel reads, the chunk-slot
// numbering of that workspace, and the tf32 operand layouts of the
// shared-memory tiles.
//
// The chunked form evaluates the token recurrence of [VA] "非连续 KV Cache" §6
// (per token S' = a S (I - b k k^T) + b v k^T, o = S' q) 64 tokens at a time.
// For one chunk (tokens 0..C-1, gates a_t, b_t) and state S (dv x dk):
//   Gam(j,t) = a_(j+1) ... a_t,  E_t = a_0 ... a_t,  F_j = Gam(j, C-1)
//   A_tj = b_t Gam(j,t) k_t.k_j (j < t),  T = (I + A)^-1,  T' = T diag(b)
//   B_tj = Gam(j,t) q_t.k_j (j <= t)
// The preparation kernel forms T', B, E, F and e_last = E_(C-1) from k, q and
// the gates alone (no state).  The state kernel then runs, per chunk,
//   P' = S (E o K)^T,  R' = S (E o Q)^T,  D = (V - P') T'^T,
//   O = R' + D B^T  (o_t of every state row),  S <- e_last S + D (F o K)
// where row t of E o K is E_t k_t and V holds v_t as column t.
#pragma once

#include <stdint.h>

namespace lsc {
namespace chunk {

constexpr int kC = 64;    // tokens per chunk
constexpr int kDK = 128;  // head_k_dim of the chunked form

// ---- workspace record of one (chunk slot, v head), fp32 --------------------
// T'[t][j] and B[t][j], 64 x 64, by 16-byte column groups: the four entries
// (t, 4 g .. 4 g + 3) at float offset rec_off(t, 4 g) = (64 g + t) * 4, so a
// warp reaching 32 consecutive rows of one group touches 512 contiguous bytes.
// Only the groups with 4 g < 4 floor(t/4) + 4 are written (the entries with
// j > t inside the last one are zero); the others are never read.
constexpr int kRecT = 0;
constexpr int kRecB = kC * kC;
constexpr int kRecE = 2 * kC * kC;     // E_t
constexpr int kRecF = kRecE + kC;      // F_t
constexpr int kRecMisc = kRecF + kC;   // [0] = e_last
constexpr int kRecFloats = kRecMisc + 16;
constexpr int64_t kRecBytes = (int64_t)kRecFloats * 4;
static_assert(kRecBytes % 16 == 0, "records keep 16-byte alignment");

// Number of 16-byte groups of row t that carry T' or B entries.
__host__ __device__ constexpr int row_groups(int t) { return t / 4 + 1; }
// Float offset of entries (t, j4 .. j4 + 3), j4 a multiple of 4.
__host__ __device__ constexpr int rec_off(int t, int j4) { return (kC * (j4 / 4) + t) * 4; }

// Chunk slots: chunk c of sequence i (tokens cu[i] + 64 c ..) has slot
// floor(cu[i] / 64) + i + c.  For cu non-decreasing in [0, T] the slots of
// different sequences never coincide and all lie below n_slots(T, n_seq).
__host__ __device__ constexpr int64_t n_slots(int64_t total_tokens, int64_t n_seq) {
  return (total_tokens + kC - 1) / kC + n_seq;
}
__host__ __device__ constexpr int64_t slot_base(int32_t cu_i, int32_t i) { return (int64_t)(cu_i / kC) + i; }
__host__ __device__ constexpr int64_t workspace_bytes(int64_t total_tokens, int64_t n_seq, int64_t Hv) {
  return n_slots(total_tokens, n_seq) * Hv * kRecBytes;
}

// ---- shared-memory tf32 operand tiles (no swizzle, 8 x 16-byte core
// matrices; see lsc_tc.h) --------------------------------------------------------
// Token-major [K; Q] tile, 128 rows x 128 channels: element (row i, channel c)
// at (i/8)*kKqRg + (c/4)*128 + (i%8)*16 + (c%4)*4 -- K-major, LBO 128, SBO kKqRg.
constexpr uint32_t kKqRg = 4096 + 16;
constexpr uint32_t kKqBytes = 16 * kKqRg;
constexpr uint32_t kQRow0 = 8 * kKqRg;  // rows 64.. (the q half)
// 64-column tiles (T', B: row t, column j; F o K: channel c, token j):
// element (row, col) at (row/8)*kRg64 + (col/4)*kLbo + (row%8)*16 + (col%4)*4
// -- K-major, LBO kLbo, SBO kRg64.
constexpr uint32_t kLbo = 128 + 16;
constexpr uint32_t kRg64 = 16 * kLbo;
constexpr uint32_t kKtBytes = 16 * kRg64;  // 128 channel rows
constexpr uint32_t kSqBytes = 8 * kRg64;   // 64 rows
static_assert(kSqBytes <= kQRow0, "a 64 x 64 tile fits over one half of the [K; Q] tile");
// The 16 bytes beyond each 4096 (resp. 128) spread the producers' 16-byte
// stores over all banks.

__host__ __device__ constexpr uint32_t kq_off(int row, int col) {
  return (uint32_t)(row / 8) * kKqRg + (uint32_t)(col / 4) * 128 + (uint32_t)(row % 8) * 16 + (uint32_t)(col % 4) * 4;
}
__host__ __device__ constexpr uint32_t sq_off(int row, int col) {
  return (uint32_t)(row / 8) * kRg64 + (uint32_t)(col / 4) * kLbo + (uint32_t)(row % 8) * 16 + (uint32_t)(col % 4) * 4;
}

}  // namespace chunk
}  // namespace lsc
