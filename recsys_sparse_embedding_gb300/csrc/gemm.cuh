// The backward's matrix products, as this library's own kernels: D = A B^T
// with both operands K-major ("TN"), fp32 results.
//
//   bf16 operands: tcgen05 MMA (kind::f16, fp32 accumulation in tensor
//   memory), 256 threads per CTA, a 128-row tile of D with the whole N
//   (<= 256) in one accumulator. Two kernels:
//   - B resident (K <= 256, no split: the products with a weight matrix):
//     persistent CTAs, one per SM, hold B in shared memory (K-major, 128-byte
//     swizzle) and walk the row tiles of A; the next tile's A loads while the
//     current tile's epilogue runs;
//   - streaming (split-K): a three-stage ring of 64-wide K-blocks of A and B.
//   Operands arrive by cp.async from all threads; one thread issues the MMAs
//   and commits them to an mbarrier. In the epilogue each warp reads 32 rows
//   of the accumulator from tensor memory (one row per lane), applies the
//   ReLU or the mask of the backward (Epi) and stores whole row segments
//   through a per-warp staging block in shared memory.
//   fp32 operands (the check mode): CUDA-core tiles of 64 x 64.
//
// Both take split-K: split z covers K-range [z * k_per_split, ...) and writes
// its partial product to D + z * split_stride; reduce() then adds the
// splits in a fixed order (deterministic).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace dsf {
namespace gemm {

// What the bf16 kernel's epilogue writes (the fp32 kernel: kEpiF32 only).
enum Epi {
  kEpiF32 = 0,       // D = A B^T (fp32)
  kEpiReluBias = 1,  // H = bf16(ReLU(A B^T + bias)) and its transpose HT;
                     // mask (nullable): bit n % 32 of word n / 32 of row m
                     // set where H[m][n] > 0
  kEpiMask = 2,      // D = A B^T; v = D where mask's bit is set, else 0;
                     // H = bf16(v) and HT; part[4 tile + j][n] = the column
                     // sums of v over rows 32 j .. 32 j + 31 of 128-row tile
                     // `tile`
  kEpiDsDq = 3,      // the dx product of the DIN backward, B's rows permuted
                     // so that columns 4d .. 4d + 3 are (dx_q, dx_s, dx_d,
                     // dx_p) of dim d: for rows m < *nvalid, ds[m][d] +=
                     // dx_s - dx_d + dx_p q and dqc[m][d] = dx_q + dx_d +
                     // dx_p s[m][d] (q: the pooled query slice of row m's
                     // sample); D is not written
};

struct TnArgs {
  const void* A;      // [M][K] (row stride lda elements), bf16 or fp32
  long long lda;
  const void* B;      // [N][K] (row stride ldb elements)
  long long ldb;
  float* D;           // [M][N] (row stride ldd), per split at D + z * split_stride;
                      // 16-byte aligned, ldd and split_stride multiples of 4
  long long ldd;
  long long M;
  int N;              // a multiple of 16 (larger N runs in chunks of 256; kEpiF32 only)
  long long K;
  long long k_per_split;  // a multiple of 64
  long long split_stride;
  int* status;        // DSF_FLAG_TIMEOUT on a wait that ran out (nullable)
  int epi;            // Epi (bf16 only)
  const float* bias;  // kEpiReluBias: [N], 16-byte aligned
  void* H;            // bf16 [M][ldh], 16-byte aligned, ldh a multiple of 8
  long long ldh;
  uint32_t* mask;     // [M][ldm] words (ldm >= N / 32): written by kEpiReluBias
                      // (nullable), read by kEpiMask
  long long ldm;
  void* HT;           // bf16 [N][ldt] (nullable): element (m, n) at n * ldt + m; 16-byte
                      // aligned, ldt a multiple of 8 and >= M rounded up to 8
                      // (entries M .. that bound of each row are overwritten)
  long long ldt;
  float* part;        // kEpiMask: [4 x M tiles][N]
  // kEpiDsDq (N = 4 Q): Q = 3 x dim
  const long long* nvalid;  // valid rows (device)
  const int* samp;          // [M] row -> sample
  const float* S;           // [M][Q] s
  float* dS;                // [M][Q] ds, updated in place
  float* dqc;               // [M][Q] out: the row's dq term
  const float* pooled;      // [B][pooled_ld]
  int pooled_ld, dim;
  int qoff[3];              // pooled column of the query slice of part k of s
};

// Launches D = A B^T over `splits` K-splits on `stream`. bf16 selects the
// operand type. Returns false if the shape is unsupported or a launch fails.
// Rows of A / B must start 16-byte aligned (lda, ldb multiples of 8 bf16 or
// 4 fp32 elements; A, B 16-byte aligned).
bool tn(const TnArgs& a, int splits, bool bf16, cudaStream_t stream);

// D (+ split z) = A^T B in bf16 over `splits` K-splits, both operands stored
// one row per K index: A [K][M] (row stride lda >= M), B [K][N] (ldb >= N), 16-byte
// aligned, strides multiples of 8 elements; fp32 results at D + z *
// split_stride, [M][ldd] (16-byte aligned, ldd and split_stride multiples of
// 4). K = 0 writes zeros. Returns false if the shape is unsupported or a
// launch fails.
bool atb(const TnArgs& a, int splits, cudaStream_t stream);

// Two independent atb products (N <= 256 each) in one launch; other shapes
// run as two atb calls.
bool atb2(const TnArgs& a0, int splits0, const TnArgs& a1, int splits1, cudaStream_t stream);

// D[m][n] = sum over s of P[s][m][n] (row strides ldp / ldd, split stride
// split_stride), in a fixed order: eight interleaved groups of splits
// (z mod 8), each summed in increasing z, then the groups in order.
bool reduce(const float* P, long long split_stride, int splits, long long ldp, float* D, long long ldd,
            long long M, int N, cudaStream_t stream);

// Two reductions as above in one launch (P1 null: the first alone).
bool reduce2(const float* P0, long long split_stride0, int splits0, long long ldp0, float* D0, long long ldd0,
             long long M0, int N0, const float* P1, long long split_stride1, int splits1, long long ldp1, float* D1,
             long long ldd1, long long M1, int N1, cudaStream_t stream);

// out[c][r] = in[r][c] for r < rows, c < cols (element size 2 or 4 bytes);
// row strides ld_in / ld_out in elements.
bool transpose(const void* in, long long ld_in, long long rows, int cols, void* out, long long ld_out, int esize,
               cudaStream_t stream);


}  // namespace gemm
}  // namespace dsf
