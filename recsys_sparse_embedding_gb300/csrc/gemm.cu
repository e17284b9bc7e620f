// The backward's matrix products (see gemm.cuh).
#include "gemm.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "dinsparse.h"
#include "ptx.cuh"

namespace dsf {
namespace gemm {
namespace {

constexpr int kWarps = 16, kThreads = 32 * kWarps;  // four warps per tensor-memory lane quarter
constexpr int kBM = 128, kBK = 64, kStages = 3;
constexpr int kStgBytes = 32 * 64;  // a warp's epilogue staging: 32 rows x 64 bytes
constexpr int kMaxGridY = 65535;

__device__ __forceinline__ void set_flag(int* status, int bits) {
  if (status && bits) atomicOr(status, bits);
}

template <int BN>
struct Tile {
  static constexpr int A_BYTES = kBM * 128;  // a 128 x 64 bf16 K-block
  static constexpr int B_BYTES = BN * 128;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int EPI_BYTES = kWarps * kStgBytes;  // the epilogue's staging
  static constexpr int BODY = kStages * STAGE > EPI_BYTES ? kStages * STAGE : EPI_BYTES;
  static constexpr int SMEM = BODY + 1024;  // + alignment slack
  static constexpr uint32_t TCOLS = BN <= 64 ? 64 : (BN <= 128 ? 128 : 256);
  static_assert(BN % 64 == 0 && BN <= 256, "tcgen05 N for M = 128, whole 16-column chunks per warp group");
  static_assert(STAGE % 1024 == 0, "stages keep the 1024-byte swizzle-atom alignment");
};

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Staging offsets (bytes) of 16-byte slot k of row r in a warp's block:
// fp32 rows of 64 bytes (4 slots), bf16 rows of 32 bytes (2 slots, 32 bytes
// of padding after every 8 rows). The slot is XOR-swizzled by row so that 8
// lanes storing one slot of 8 rows, and 8 lanes loading whole rows, each
// touch 8 different bank groups; the padding puts rows r and r + 8 (read
// together by the transposed copy) in different bank groups.
__device__ __forceinline__ int stg32(int r, int k) { return r * 64 + ((k ^ ((r >> 1) & 3)) << 4); }
__device__ __forceinline__ int stg16(int r, int k) { return r * 32 + (r >> 3) * 32 + ((k ^ ((r >> 2) & 1)) << 4); }

// The epilogue of one 128-row tile whose accumulator (BN columns) starts at
// tensor-memory column tbase. Warp w reads rows 32 (w % 4) .. + 31 (its lane
// quarter of tensor memory), one row per lane, over the 16-column chunks
// w / 4, w / 4 + 4, ... Every output goes through the warp's staging block
// in shared memory, so that each store instruction writes whole 32-byte
// sectors: D (fp32) and H (bf16) as row segments, HT (H transposed) as
// 16-row column segments. Column sums (kEpiMask) add down the staged block
// (rows 0-15 and 16-31 in two lanes, then the two) and go out per lane
// quarter. This call covers columns n0 .. n0 + W - 1 of the tile, whose
// accumulator starts at tensor-memory column tcol. E: kWarps staging blocks.
// have_acc false: the product is zero.
// bias: kEpiReluBias's bias (global or shared). mpre >= 0: the chunk's mask
// bits, loaded by the caller (kEpiMask, one chunk per warp). work false:
// nothing (a run that gave up).
template <int BN, int W, int EPI = -1>
__device__ __forceinline__ void epilogue(const TnArgs& a, uint8_t* E, uint32_t tcol, long long m0, int n0,
                                         long long tile, float* D, bool have_acc, const float* bias = nullptr,
                                         long long mpre = -1, bool work = true) {
  const int epi = EPI >= 0 ? EPI : a.epi;  // (compile-time where the caller knows it)
  constexpr int NCH = W / 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = warp & 3, grp = warp >> 2;
  uint8_t* stg = E + warp * kStgBytes;
  const long long rbase = m0 + q * 32, row = rbase + lane;
  const bool live = row < a.M;
  __nv_bfloat16* H = static_cast<__nv_bfloat16*>(a.H);
  uint16_t* HT = static_cast<uint16_t*>(a.HT);
  uint16_t* mrow = a.mask ? reinterpret_cast<uint16_t*>(a.mask + (live ? row : 0) * a.ldm) : nullptr;
  long long ds_rows = 0;  // kEpiDsDq: rows below this are valid
  if (epi == kEpiDsDq) {
    const long long nv = __ldg(a.nvalid);
    ds_rows = nv < a.M ? nv : a.M;
  }
#pragma unroll
  for (int ch = grp; ch < NCH; ch += 4) {
    const int c0 = n0 + ch * 16;
    if (c0 >= a.N || !work) break;
    const uint32_t mbits =
        mpre >= 0 ? uint32_t(mpre) : ((epi == kEpiMask && live) ? uint32_t(mrow[c0 >> 4]) : 0u);  // (before the wait below)
    // kEpiDsDq: the row's sample, s and ds for dims c0 / 4 .. + 3 (before the wait below)
    int ds_samp = 0;
    float4 ds_s = make_float4(0.f, 0.f, 0.f, 0.f), ds_d = ds_s;
    if (epi == kEpiDsDq && row < ds_rows) {
      ds_samp = __ldg(a.samp + row);
      ds_s = __ldg(reinterpret_cast<const float4*>(a.S + row * (a.N / 4) + (c0 >> 2)));
      ds_d = *reinterpret_cast<const float4*>(a.dS + row * (a.N / 4) + (c0 >> 2));
    }
    float v[16];
    if (have_acc) {
      tmem_ld16(tcol + (uint32_t(q * 32) << 16) + uint32_t(ch * 16), v);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0.f;
    }
    if (D) {  // fp32: 64-byte row segments
#pragma unroll
      for (int k = 0; k < 4; ++k)
        *reinterpret_cast<float4*>(stg + stg32(lane, k)) = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
      __syncwarp();
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int r = it * 8 + (lane >> 2), k = lane & 3;
        const long long gr = rbase + r;
        if (gr < a.M && c0 + 4 * k < a.N)
          *reinterpret_cast<float4*>(D + gr * a.ldd + c0 + 4 * k) = *reinterpret_cast<const float4*>(stg + stg32(r, k));
      }
      __syncwarp();
    }
    if (epi == kEpiF32) continue;
    if (epi == kEpiDsDq) {
      // columns c0 .. c0 + 15: dims d0 .. d0 + 3, four columns each
      const int d0 = c0 >> 2;
      if (row < ds_rows) {
        const int part = d0 / a.dim, e = d0 - part * a.dim;
        const float4 q4 = __ldg(reinterpret_cast<const float4*>(a.pooled + (long long)ds_samp * a.pooled_ld +
                                                                a.qoff[part] + e));
        const float qv[4] = {q4.x, q4.y, q4.z, q4.w}, sv[4] = {ds_s.x, ds_s.y, ds_s.z, ds_s.w};
        const float dv[4] = {ds_d.x, ds_d.y, ds_d.z, ds_d.w};
        float o[4], g[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float xq = v[4 * t], xs = v[4 * t + 1], xd = v[4 * t + 2], xp = v[4 * t + 3];
          o[t] = dv[t] + xs - xd + xp * qv[t];
          g[t] = xq + xd + xp * sv[t];
        }
        *reinterpret_cast<float4*>(a.dS + row * (a.N / 4) + d0) = make_float4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<float4*>(a.dqc + row * (a.N / 4) + d0) = make_float4(g[0], g[1], g[2], g[3]);
      }
      continue;
    }
    if (epi == kEpiReluBias) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 b = reinterpret_cast<const float4*>((bias ? bias : a.bias) + c0)[k];
        v[4 * k] = fmaxf(v[4 * k] + b.x, 0.f);
        v[4 * k + 1] = fmaxf(v[4 * k + 1] + b.y, 0.f);
        v[4 * k + 2] = fmaxf(v[4 * k + 2] + b.z, 0.f);
        v[4 * k + 3] = fmaxf(v[4 * k + 3] + b.w, 0.f);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (!((mbits >> j) & 1u)) v[j] = 0.f;
    }
    uint32_t p[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) p[t] = bf16x2(v[2 * t], v[2 * t + 1]);
    if (epi == kEpiReluBias && mrow && live) {
      // bit j: bf16 value j is > 0 (ReLU outputs are >= 0 or -0); a half h
      // of x = p & 0x7fff7fff is nonzero iff h + 0x7fff carries into its
      // top bit
      uint32_t bits = 0;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const uint32_t y = (p[t] & 0x7fff7fffu) + 0x7fff7fffu;
        bits |= ((y >> 15) & 1u) << (2 * t) | (y >> 31) << (2 * t + 1);
      }
      mrow[c0 >> 4] = uint16_t(bits);
    }
    // bf16: 32-byte row segments, then 16-row segments of HT's rows
#pragma unroll
    for (int k = 0; k < 2; ++k)
      *reinterpret_cast<uint4*>(stg + stg16(lane, k)) = make_uint4(p[4 * k], p[4 * k + 1], p[4 * k + 2], p[4 * k + 3]);
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int r = it * 16 + (lane >> 1), k = lane & 1;
      const long long gr = rbase + r;
      if (gr < a.M && c0 + 8 * k < a.N)
        *reinterpret_cast<uint4*>(H + gr * a.ldh + c0 + 8 * k) = *reinterpret_cast<const uint4*>(stg + stg16(r, k));
    }
    if (HT) {
      // lane pair (2j, 2j + 1): column j, rows 8 (2i + hb) .. + 7 of the
      // block (one 32-byte sector of HT's row per lane pair)
      const int j = lane >> 1, hb = lane & 1;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r0 = 16 * i + 8 * hb;
        uint16_t e[8];
#pragma unroll
        for (int t = 0; t < 8; ++t)
          e[t] = *reinterpret_cast<const uint16_t*>(stg + stg16(r0 + t, j >> 3) + ((j & 7) << 1));
        if (rbase + r0 < a.M && c0 + j < a.N)
          *reinterpret_cast<uint4*>(HT + (long long)(c0 + j) * a.ldt + rbase + r0) =
              make_uint4(uint32_t(e[0]) | uint32_t(e[1]) << 16, uint32_t(e[2]) | uint32_t(e[3]) << 16,
                         uint32_t(e[4]) | uint32_t(e[5]) << 16, uint32_t(e[6]) | uint32_t(e[7]) << 16);
      }
    }
    __syncwarp();
    if (epi == kEpiMask && a.part) {
      // the masked fp32 block; lane l adds column l % 16 down rows
      // 16 (l / 16) .. + 15 (the upper lanes rotated by one row: another
      // bank group), then the lower lane adds the upper lane's sum and
      // stores the column sum of the warp's 32 rows
#pragma unroll
      for (int k = 0; k < 4; ++k)
        *reinterpret_cast<float4*>(stg + stg32(lane, k)) = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
      __syncwarp();
      const int c = lane & 15, hb = lane >> 4;
      float sum = 0.f;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int rr = 16 * hb + ((t + hb) & 15);
        sum += *reinterpret_cast<const float*>(stg + stg32(rr, c >> 2) + ((c & 3) << 2));
      }
      sum += __shfl_down_sync(0xffffffffu, sum, 16);
      if (lane < 16 && c0 + lane < a.N) a.part[(tile * 4 + q) * a.N + c0 + lane] = sum;
      __syncwarp();
    }
  }
}

// D (+ split) = A[m0 : m0 + 128][k-range] * B[0 : BN][k-range]^T, bf16, with
// the epilogue a.epi.
template <int BN>
__global__ void __launch_bounds__(kThreads, 1) tn_bf16_kernel(const TnArgs a) {
  using T = Tile<BN>;
  extern __shared__ uint8_t dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar[kStages];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_;
  const int tid = threadIdx.x, warp = tid >> 5;
  const long long m0 = (long long)blockIdx.x * kBM;
  const long long k0 = (long long)blockIdx.y * a.k_per_split;
  const long long k1 = k0 + a.k_per_split < a.K ? k0 + a.k_per_split : a.K;
  const int nkb = k1 > k0 ? int((k1 - k0 + kBK - 1) / kBK) : 0;
  float* D = a.D ? a.D + (long long)blockIdx.y * a.split_stride : nullptr;
  const __nv_bfloat16* A = static_cast<const __nv_bfloat16*>(a.A);
  const __nv_bfloat16* Bm = static_cast<const __nv_bfloat16*>(a.B);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
    fence_mbarrier_init();
    abort_ = 0;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, T::TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;

  // K-block kb into its stage: 16-byte chunks in the 128-byte swizzle layout
  // (chunk c of row r at r * 128 + (c ^ (r % 8)) * 16); rows past M or N and
  // elements past the split's K-range are zero-filled.
  auto load = [&](int kb) {
    uint8_t* sa = sm + (kb % kStages) * T::STAGE;
    uint8_t* sb = sa + T::A_BYTES;
    const long long kk = k0 + (long long)kb * kBK;
    for (int q = tid; q < kBM * 8; q += kThreads) {
      const int r = q >> 3, c = q & 7;
      const long long row = m0 + r, k = kk + c * 8;
      long long v = row < a.M ? k1 - k : 0;
      v = v < 0 ? 0 : (v > 8 ? 8 : v);
      const __nv_bfloat16* src = v > 0 ? A + row * a.lda + k : A;
      cp_async_16_ca(sa + r * 128 + ((c ^ (r & 7)) << 4), src, uint32_t(v * 2));
    }
    for (int q = tid; q < BN * 8; q += kThreads) {
      const int r = q >> 3, c = q & 7;
      const long long k = kk + c * 8;
      long long v = r < a.N ? k1 - k : 0;
      v = v < 0 ? 0 : (v > 8 ? 8 : v);
      const __nv_bfloat16* src = v > 0 ? Bm + (long long)r * a.ldb + k : Bm;
      cp_async_16_ca(sb + r * 128 + ((c ^ (r & 7)) << 4), src, uint32_t(v * 2));
    }
  };
  constexpr uint32_t IDESC = idesc_bf16_f32(kBM, BN);
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nkb) load(s);
    cp_async_commit();
  }
  int issued = -1;  // last K-block whose MMAs were committed
  for (int kb = 0; kb < nkb; ++kb) {
    cp_async_wait_one_pending();  // (kStages - 2 = 1 group may stay in flight)
    fence_proxy_async_smem();
    __syncthreads();
    if (abort_) break;
    if (tid == 0) {
      tc_fence_after();
      const uint32_t sa = smem_u32(sm + (kb % kStages) * T::STAGE), sb = sa + T::A_BYTES;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        tc_mma_f16(tbase, sw128_kmajor_desc(sa + kk * 32), sw128_kmajor_desc(sb + kk * 32), IDESC,
                   (kb > 0 || kk > 0) ? 1u : 0u);
      tc_commit(&bar[kb % kStages]);
    }
    issued = kb;
    // block kb + kStages - 1 goes into the stage block kb - 1 used: wait for
    // that block's MMAs first (block kb's run meanwhile)
    const int nx = kb + kStages - 1;
    if (nx < nkb) {
      if (kb >= 1) {
        if (tid == 0 && !mbar_wait(&bar[(kb - 1) % kStages], uint32_t(((kb - 1) / kStages) & 1))) abort_ = 1;
        __syncthreads();
      }
      if (!abort_) load(nx);
    }
    cp_async_commit();
  }
  cp_async_wait_all();
  // every MMA done (a commit tracks all earlier MMAs of its thread)
  if (tid == 0 && issued >= 0 && !mbar_wait(&bar[issued % kStages], uint32_t((issued / kStages) & 1))) abort_ = 1;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!abort_) epilogue<BN, BN>(a, sm, tbase, m0, 0, blockIdx.x, D, nkb > 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, T::TCOLS);
  if (tid == 0 && abort_) set_flag(a.status, DSF_FLAG_TIMEOUT);
}

// B resident: D = A B^T with N <= 256 and K <= 64 * KB <= 256 (B, the MLP
// weights, fits shared memory whole). Work units of 128 rows x 64 columns
// (unit u: row tile u / NU, columns 64 (u % NU) ..), NU = BN / 64 per tile;
// persistent CTAs, one per SM, each take a contiguous run of units (runs
// differ by at most one unit; a row tile's A is loaded once per CTA that
// touches it). Warp-specialised: warp kWarps loads A and issues the MMAs
// (one thread) into two 64-column accumulators in tensor memory; warps
// 0 .. kWarps - 1 run the epilogue. They hand over through mbarriers:
// full[b] (the unit's MMAs committed) and empty[b] (every epilogue warp has
// read accumulator b), so the MMAs and A loads of later units overlap the
// epilogue of earlier ones and the epilogue warps never wait for each other.
template <int BN, int KB>
struct RTile {
  static constexpr int UN = 64;  // columns per work unit
  static constexpr int NU = BN / UN;
  static constexpr int B_BYTES = KB * BN * 128;
  static constexpr int A_BYTES = KB * kBM * 128;
  static constexpr int E_BYTES = kWarps * kStgBytes;
  static constexpr int BIAS_BYTES = BN * 4;
  static constexpr int SMEM = B_BYTES + A_BYTES + E_BYTES + BIAS_BYTES + 1024;
  static constexpr uint32_t TCOLS = 2 * UN;
  static_assert(B_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "1024-byte swizzle-atom alignment");
  static_assert(BN % UN == 0 && BN <= 256 && UN == 4 * 16, "one 16-column chunk per epilogue warp and unit");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

template <int BN, int KB, int EPI>
__global__ void __launch_bounds__(kThreads + 32, 1)
    tn_bf16_resident_kernel(const TnArgs a, const __grid_constant__ CUtensorMap mapA,
                            const __grid_constant__ CUtensorMap mapB) {
  using T = RTile<BN, KB>;
  constexpr int UN = T::UN, NU = T::NU;
  constexpr uint32_t A_TX = KB * kBM * 128, B_TX = KB * BN * 128;
  extern __shared__ uint8_t dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = sm;
  uint8_t* sA = sm + T::B_BYTES;
  uint8_t* sE = sA + T::A_BYTES;
  float* sBias = reinterpret_cast<float*>(sE + T::E_BYTES);
  __shared__ uint64_t full[2], empty[2], abar, bbar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long tiles = (a.M + kBM - 1) / kBM;
  const long long units = tiles * NU;
  const long long u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
  if (u0 >= u1) return;
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], kWarps);
    }
    mbar_init(&abar, 1);
    mbar_init(&bbar, 1);
    fence_mbarrier_init();
    abort_ = 0;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, T::TCOLS);
    tmem_relinquish();
  }
  if (EPI == kEpiReluBias)
    for (int c = tid; c < BN; c += blockDim.x) sBias[c] = c < a.N ? a.bias[c] : 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;

  if (warp == kWarps) {
    // ------------------------------------------------ producer (one thread):
    // TMA loads of B (once) and of each row tile's A, MMAs of every unit
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(kBM, UN);
      uint32_t inflight = 0;             // accumulators with a commit not yet waited for
      long long last0 = -1, last1 = -1;  // the last unit committed to full[0] / full[1]
      uint32_t na = 0;                   // A loads issued (abar's phases)
      bool a_pending = false, ok = true;
      mbar_arrive_expect_tx(&bbar, B_TX);
      for (int kb = 0; kb < KB; ++kb) tma_load_2d(sB + kb * (BN * 128), &mapB, kb * kBK, 0, &bbar);
      auto load_a = [&](long long t) {
        mbar_arrive_expect_tx(&abar, A_TX);
        for (int kb = 0; kb < KB; ++kb) tma_load_2d(sA + kb * (kBM * 128), &mapA, kb * kBK, int(t * kBM), &abar);
        ++na;
        a_pending = true;
      };
      load_a(u0 / NU);
      ok = mbar_wait(&bbar, 0);
      for (long long u = u0; u < u1 && ok; ++u) {
        const int b = int(u & 1);
        const long long k = u - u0;
        if (a_pending) {
          if (!(ok = mbar_wait(&abar, (na - 1) & 1u))) break;
          a_pending = false;
        }
        if (k >= 2 && !(ok = mbar_wait(&empty[b], uint32_t(((k - 2) >> 1) & 1)))) break;
        tc_fence_after();
        const uint32_t d = tbase + uint32_t(b) * UN;
        const int nq = int(u % NU);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma_f16(d, sw128_kmajor_desc(smem_u32(sA + kb * (kBM * 128)) + kk * 32),
                       sw128_kmajor_desc(smem_u32(sB + kb * (BN * 128) + nq * (UN * 128)) + kk * 32), IDESC,
                       (kb > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&full[b]);
        inflight |= 1u << b;
        (b ? last1 : last0) = u;
        if (u + 1 < u1 && (u + 1) % NU == 0) {
          // the next unit starts a row tile: its A loads once this unit's MMAs
          // (the last readers of the current A) are done
          if (!(ok = mbar_wait(&full[b], uint32_t((k >> 1) & 1)))) break;
          load_a((u + 1) / NU);
        }
      }
      if (!ok) {
        atomicExch(&abort_, 1);
        // (copies and MMAs that may still run: wait, bounded, before the
        // buffers and accumulators are released)
        if (a_pending) mbar_wait(&abar, (na - 1) & 1u);
        if ((inflight & 1u) && last0 >= 0) mbar_wait(&full[0], uint32_t(((last0 - u0) >> 1) & 1));
        if ((inflight & 2u) && last1 >= 0) mbar_wait(&full[1], uint32_t(((last1 - u0) >> 1) & 1));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue warps
    const int q = warp & 3, grp = warp >> 2;
    // the mask bits of this warp's chunk in unit u (kEpiMask), loaded a unit ahead
    auto mask_of = [&](long long u) -> long long {
      if (EPI != kEpiMask || u >= u1) return 0;
      const long long row = (u / NU) * kBM + q * 32 + lane;
      const int c0 = int(u % NU) * UN + grp * 16;
      return (row < a.M && c0 < a.N) ? (long long)reinterpret_cast<const uint16_t*>(a.mask + row * a.ldm)[c0 >> 4]
                                     : 0;
    };
    long long mnext = mask_of(u0);
    for (long long u = u0; u < u1; ++u) {
      const int b = int(u & 1);
      const long long k = u - u0;
      bool ok = !*reinterpret_cast<volatile int*>(&abort_);
      if (ok && lane == 0) ok = mbar_wait(&full[b], uint32_t((k >> 1) & 1));
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok && lane == 0) atomicExch(&abort_, 1);
      tc_fence_after();
      const long long mcur = mnext;
      mnext = mask_of(u + 1);
      epilogue<BN, UN, EPI>(a, sE, tbase + uint32_t(b) * UN, (u / NU) * kBM, int(u % NU) * UN, u / NU, a.D, true, sBias,
                       EPI == kEpiMask ? mcur : -1, ok);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[b]);
    }
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, T::TCOLS);
  if (tid == 0 && abort_) set_flag(a.status, DSF_FLAG_TIMEOUT);
}

// D (+ split) = A^T B with both operands stored one row per K index (A
// [K][M], B [K][N]): the weight gradients' sums over positions, read from
// the activations as they are stored. A CTA computes a 128 x BN
// tile over its K-split. Operand tiles arrive by TMA as 64 x 64 boxes in the
// 128-byte swizzle (rows of 64 M- or N-elements, one row per position), which
// is the MN-major canonical layout: atoms of 8 positions x 64 elements
// (1024 bytes; SBO, along K), the next 64 elements 8 KB further (LBO, along
// M or N). One thread keeps kAStages K-blocks in flight and issues the MMAs;
// all warps run the epilogue.
constexpr int kAStages = 4;

template <int BN>
struct ATile {
  static constexpr int NB = BN / 64;
  static constexpr int A_BYTES = 2 * 8192, B_BYTES = NB * 8192, STAGE = A_BYTES + B_BYTES;
  static constexpr int SMEM = kAStages * STAGE + kWarps * kStgBytes + 1024;
  static constexpr uint32_t TCOLS = BN <= 64 ? 64 : (BN <= 128 ? 128 : 256);
  static_assert(BN % 64 == 0 && BN <= 256, "whole 64-element atoms along N");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(8192u >> 4) << 16;  // LBO: the next 64 elements along M / N
  d |= static_cast<uint64_t>(1024u >> 4) << 32;  // SBO: the next 8 positions along K
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;  // 128-byte swizzle
  return d;
}

// Up to two independent products in one launch: CTAs [0, g0) take job 0
// (mt0 row tiles x its splits, tile-minor), the rest job 1.
template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    atb_bf16_kernel(const __grid_constant__ TnArgs a0, const __grid_constant__ TnArgs a1, int g0, int mt0, int mt1,
                    const __grid_constant__ CUtensorMap mapA0, const __grid_constant__ CUtensorMap mapB0,
                    const __grid_constant__ CUtensorMap mapA1, const __grid_constant__ CUtensorMap mapB1) {
  using T = ATile<BN>;
  const bool j1 = int(blockIdx.x) >= g0;
  const TnArgs& a = j1 ? a1 : a0;
  const CUtensorMap* mapA = j1 ? &mapA1 : &mapA0;
  const CUtensorMap* mapB = j1 ? &mapB1 : &mapB0;
  const int local = int(blockIdx.x) - (j1 ? g0 : 0), mt = j1 ? mt1 : mt0;
  const int mtile = local % mt, split = local / mt;
  extern __shared__ uint8_t dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sE = sm + kAStages * T::STAGE;
  __shared__ uint64_t full[kAStages], done[kAStages];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_;
  const int tid = threadIdx.x, warp = tid >> 5;
  const long long m0 = (long long)mtile * kBM;
  const long long k0 = (long long)split * a.k_per_split;
  const long long k1 = k0 + a.k_per_split < a.K ? k0 + a.k_per_split : a.K;
  const int nkb = k1 > k0 ? int((k1 - k0 + kBK - 1) / kBK) : 0;
  float* D = a.D + (long long)split * a.split_stride;
  if (tid == 0) {
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&done[i], 1);
    }
    fence_mbarrier_init();
    abort_ = 0;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, T::TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  if (tid == 0 && nkb > 0) {
    constexpr uint32_t IDESC = idesc_bf16_f32(kBM, BN) | (1u << 15) | (1u << 16);  // A and B MN-major
    // boxes wholly past M or N are not loaded: the accumulator rows and
    // columns they feed are never stored
    const long long mrem = a.M - m0;
    const int na = mrem > 64 ? 2 : 1, nb = int((a.N + 63) / 64) < T::NB ? int((a.N + 63) / 64) : T::NB;
    const uint32_t tx = uint32_t(na + nb) * 8192u;
    auto load = [&](int kb) {
      uint8_t* st = sm + (kb % kAStages) * T::STAGE;
      uint64_t* bar = &full[kb % kAStages];
      const int y = int(k0 + (long long)kb * kBK);
      mbar_arrive_expect_tx(bar, tx);
      for (int j = 0; j < na; ++j) tma_load_2d(st + j * 8192, mapA, int(m0) + 64 * j, y, bar);
      for (int j = 0; j < nb; ++j) tma_load_2d(st + T::A_BYTES + j * 8192, mapB, 64 * j, y, bar);
    };
    bool ok = true;
    int issued = 0;  // K-blocks whose loads were issued
    for (; issued < kAStages && issued < nkb; ++issued) load(issued);
    int last = -1;  // the last K-block whose MMAs were committed
    for (int kb = 0; kb < nkb && ok; ++kb) {
      const int st = kb % kAStages;
      const uint32_t par = uint32_t((kb / kAStages) & 1);
      if (!(ok = mbar_wait(&full[st], par))) break;
      tc_fence_after();
      const uint32_t sa = smem_u32(sm + st * T::STAGE), sb = sa + T::A_BYTES;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        tc_mma_f16(tbase, sw128_mnmajor_desc(sa + kk * 2048), sw128_mnmajor_desc(sb + kk * 2048), IDESC,
                   (kb > 0 || kk > 0) ? 1u : 0u);
      tc_commit(&done[st]);
      last = kb;
      if (issued < nkb) {
        // block `issued` reuses this stage once these MMAs are done
        if (!(ok = mbar_wait(&done[st], par))) break;
        load(issued++);
      }
    }
    // every MMA done (a commit covers all earlier MMAs of the thread); on a
    // timeout, the copies still in flight are waited for too (bounded)
    if (last >= 0) ok = mbar_wait(&done[last % kAStages], uint32_t((last / kAStages) & 1)) && ok;
    if (!ok) {
      abort_ = 1;
      for (int kb = last + 1; kb < issued; ++kb) mbar_wait(&full[kb % kAStages], uint32_t((kb / kAStages) & 1));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!abort_) epilogue<BN, BN>(a, sE, tbase, m0, 0, mtile, D, nkb > 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, T::TCOLS);
  if (tid == 0 && abort_) set_flag(a.status, DSF_FLAG_TIMEOUT);
}

// fp32 operands on the CUDA cores: 64 x 64 tiles of D, 256 threads, 4 x 4
// results each; K-steps of 16 staged in shared memory.
__global__ void __launch_bounds__(256) tn_f32_kernel(const TnArgs a, int n0) {
  constexpr int BM = 64, BN = 64, BK = 16;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const long long m0 = (long long)blockIdx.x * BM;
  const int nb = n0 + blockIdx.z * BN;
  const long long k0 = (long long)blockIdx.y * a.k_per_split;
  const long long k1 = k0 + a.k_per_split < a.K ? k0 + a.k_per_split : a.K;
  const float* A = static_cast<const float*>(a.A);
  const float* Bm = static_cast<const float*>(a.B);
  float* D = a.D + (long long)blockIdx.y * a.split_stride;
  float acc[4][4] = {};
  for (long long kk = k0; kk < k1; kk += BK) {
    // 64 rows x 16 k of A and of B: four elements per thread each
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + i * 256, r = e >> 4, c = e & 15;
      const long long k = kk + c;
      const long long ra = m0 + r;
      const int rb = nb + r;
      As[c][r] = (ra < a.M && k < k1) ? A[ra * a.lda + k] : 0.f;
      Bs[c][r] = (rb < a.N && k < k1) ? Bm[(long long)rb * a.ldb + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < BK; ++c) {
      float x[4], y[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[i] = As[c][ty * 4 + i];
        y[i] = Bs[c][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(x[i], y[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long row = m0 + ty * 4 + i;
    if (row >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = nb + tx * 4 + j;
      if (col < a.N) D[row * a.ldd + col] = acc[i][j];
    }
  }
}

// 32 consecutive outputs per block of 256 threads: warp g adds splits g,
// g + 8, g + 16, ... in increasing order (eight loads in flight), then warp
// 0 adds the eight warps' sums in warp order. The order is fixed, so the
// result is deterministic. Blocks [0, b0) take job 0, the rest job 1.
struct RedJob {
  const float* P;
  long long split_stride, ldp, ldd, M;
  float* D;
  int splits, N;
};
__global__ void __launch_bounds__(256) reduce_kernel(const RedJob j0, const RedJob j1, int b0) {
  __shared__ float part[8][33];
  const bool second = int(blockIdx.x) >= b0;
  const RedJob& J = second ? j1 : j0;
  const int nblk = second ? int(gridDim.x) - b0 : b0, blk = int(blockIdx.x) - (second ? b0 : 0);
  const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
  const long long total = J.M * J.N;
  for (long long base = blk * 32LL; base < total; base += nblk * 32LL) {
    const long long i = base + lane;
    const long long m = i < total ? i / J.N : 0;
    const int n = int(i - m * J.N);
    float s = 0.f;
    if (i < total) {
      const float* q = J.P + m * J.ldp + n;
      for (int z0 = g; z0 < J.splits; z0 += 64) {
        float v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) v[t] = z0 + 8 * t < J.splits ? q[(long long)(z0 + 8 * t) * J.split_stride] : 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t)
          if (z0 + 8 * t < J.splits) s += v[t];
      }
    }
    part[g][lane] = s;
    __syncthreads();
    if (g == 0 && i < total) {
      float r = part[0][lane];
#pragma unroll
      for (int k = 1; k < 8; ++k) r += part[k][lane];
      J.D[m * J.ldd + n] = r;
    }
    __syncthreads();
  }
}

// The same sums four outputs at a time (N, ldp, ldd and split_stride
// multiples of 4; P and D 16-byte aligned): 128 consecutive outputs per
// block, float4 loads, the same fixed order per output.
__global__ void __launch_bounds__(256) reduce4_kernel(const RedJob j0, const RedJob j1, int b0) {
  __shared__ float4 part[8][32];
  const bool second = int(blockIdx.x) >= b0;
  const RedJob& J = second ? j1 : j0;
  const int nblk = second ? int(gridDim.x) - b0 : b0, blk = int(blockIdx.x) - (second ? b0 : 0);
  const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
  const long long total4 = J.M * J.N / 4;
  for (long long base = blk * 32LL; base < total4; base += nblk * 32LL) {
    const long long i = base + lane;
    const long long m = i < total4 ? (4 * i) / J.N : 0;
    const int n = int(4 * i - m * J.N);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < total4) {
      const float* q = J.P + m * J.ldp + n;
      for (int z0 = g; z0 < J.splits; z0 += 64) {
        float4 v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t)
          v[t] = z0 + 8 * t < J.splits ? *reinterpret_cast<const float4*>(q + (long long)(z0 + 8 * t) * J.split_stride)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 8; ++t)
          if (z0 + 8 * t < J.splits) s.x += v[t].x, s.y += v[t].y, s.z += v[t].z, s.w += v[t].w;
      }
    }
    part[g][lane] = s;
    __syncthreads();
    if (g == 0 && i < total4) {
      float4 r = part[0][lane];
#pragma unroll
      for (int k = 1; k < 8; ++k) {
        const float4 x = part[k][lane];
        r.x += x.x, r.y += x.y, r.z += x.z, r.w += x.w;
      }
      *reinterpret_cast<float4*>(J.D + m * J.ldd + n) = r;
    }
    __syncthreads();
  }
}

// 2-byte elements, 64 x 64 tiles: 16-byte loads (8 consecutive columns of a
// row) and 16-byte stores (8 consecutive rows of a column); both strides
// multiples of 8 elements.
__global__ void transpose16_kernel(const uint16_t* in, long long ld_in, long long rows, int cols, uint16_t* out,
                                   long long ld_out) {
  __shared__ uint16_t t[64][64 + 2];
  const long long r0 = (long long)blockIdx.x * 64;
  const int c0 = blockIdx.y * 64;
  for (int q = threadIdx.x; q < 64 * 8; q += blockDim.x) {
    const int i = q >> 3, j = (q & 7) * 8;
    const long long r = r0 + i;
    uint16_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (r < rows) {
      if (c0 + j + 8 <= cols) {
        const uint4 x = *reinterpret_cast<const uint4*>(in + r * ld_in + c0 + j);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) { v[2 * k] = uint16_t(w[k]); v[2 * k + 1] = uint16_t(w[k] >> 16); }
      } else {
        for (int k = 0; c0 + j + k < cols && k < 8; ++k) v[k] = in[r * ld_in + c0 + j + k];
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) t[i][j + k] = v[k];
  }
  __syncthreads();
  for (int q = threadIdx.x; q < 64 * 8; q += blockDim.x) {
    const int j = q >> 3, i = (q & 7) * 8;
    const int c = c0 + j;
    const long long r = r0 + i;
    if (c >= cols || r >= rows) continue;
    if (r + 8 <= rows) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) w[k] = uint32_t(t[i + 2 * k][j]) | (uint32_t(t[i + 2 * k + 1][j]) << 16);
      *reinterpret_cast<uint4*>(out + (long long)c * ld_out + r) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      for (int k = 0; r + k < rows; ++k) out[(long long)c * ld_out + r + k] = t[i + k][j];
    }
  }
}

template <typename E>
__global__ void transpose_kernel(const E* in, long long ld_in, long long rows, int cols, E* out, long long ld_out) {
  __shared__ E t[32][33];
  const long long r0 = (long long)blockIdx.x * 32;
  const int c0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const long long r = r0 + i;
    const int c = c0 + threadIdx.x;
    if (r < rows && c < cols) t[i][threadIdx.x] = in[r * ld_in + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i;
    const long long r = r0 + threadIdx.x;
    if (r < rows && c < cols) out[(long long)c * ld_out + r] = t[threadIdx.x][i];
  }
}

template <int BN>
bool launch_bf16(const TnArgs& a, int splits, cudaStream_t s) {
  using T = Tile<BN>;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(tn_bf16_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM) !=
        cudaSuccess)
      return false;
    attr_set[dev] = true;
  }
  const long long mt = (a.M + kBM - 1) / kBM;
  if (mt <= 0 || mt > 0x7fffffff || splits < 1 || splits > kMaxGridY) return false;
  tn_bf16_kernel<BN><<<dim3(unsigned(mt), unsigned(splits)), kThreads, T::SMEM, s>>>(a);
  return cudaGetLastError() == cudaSuccess;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A 2-D bf16 tensor map over rows x cols (row stride ld elements) whose box is
// 64 columns (128 bytes, the 128-byte swizzle span) by box_rows rows; reads
// past the tensor's edge fill with zeros.
bool tensor_map(CUtensorMap* m, const void* base, long long rows, long long cols, long long ld, int box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_tiled();
  if (!fn || rows <= 0 || cols <= 0 || box_rows <= 0 || box_rows > 256) return false;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(ld) * 2};
  const cuuint32_t box[2] = {cuuint32_t(kBK), cuuint32_t(box_rows)};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int KB, int EPI>
int launch_resident_e(const TnArgs& a, cudaStream_t s) {  // 1 ok, 0 failed
  using T = RTile<BN, KB>;
  static bool attr_set[64] = {};
  static int nsm[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(tn_bf16_resident_kernel<BN, KB, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&nsm[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    attr_set[dev] = true;
  }
  const long long units = (a.M + kBM - 1) / kBM * T::NU;
  const long long g = units < nsm[dev] ? units : nsm[dev];
  if (g <= 0) return 1;
  CUtensorMap mapA, mapB;
  if (!tensor_map(&mapA, a.A, a.M, a.K, a.lda, kBM) || !tensor_map(&mapB, a.B, a.N, a.K, a.ldb, BN)) return 0;
  tn_bf16_resident_kernel<BN, KB, EPI><<<unsigned(g), kThreads + 32, T::SMEM, s>>>(a, mapA, mapB);
  return cudaGetLastError() == cudaSuccess ? 1 : 0;
}

template <int BN, int KB>
int launch_resident(const TnArgs& a, cudaStream_t s) {  // 1 ok, 0 failed
  switch (a.epi) {
    case kEpiF32: return launch_resident_e<BN, KB, kEpiF32>(a, s);
    case kEpiReluBias: return launch_resident_e<BN, KB, kEpiReluBias>(a, s);
    case kEpiMask: return launch_resident_e<BN, KB, kEpiMask>(a, s);
    case kEpiDsDq: return launch_resident_e<BN, KB, kEpiDsDq>(a, s);
    default: return 0;
  }
}

// Job 1 (a1 non-null) runs in the same launch as job 0.
template <int BN>
bool launch_atb(const TnArgs& a0, int s0, const TnArgs* a1, int s1, cudaStream_t s) {
  using T = ATile<BN>;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(atb_bf16_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM) != cudaSuccess)
      return false;
    attr_set[dev] = true;
  }
  const long long mt0 = (a0.M + kBM - 1) / kBM, mt1 = a1 ? (a1->M + kBM - 1) / kBM : 1;
  const long long g0 = mt0 * s0, g1 = a1 ? mt1 * s1 : 0;
  if (mt0 <= 0 || mt1 <= 0 || s0 < 1 || (a1 && s1 < 1) || g0 + g1 > 0x7fffffff) return false;
  CUtensorMap mA0, mB0, mA1, mB1;
  if (!tensor_map(&mA0, a0.A, a0.K, a0.M, a0.lda, 64) || !tensor_map(&mB0, a0.B, a0.K, a0.N, a0.ldb, 64)) return false;
  if (a1) {
    if (!tensor_map(&mA1, a1->A, a1->K, a1->M, a1->lda, 64) || !tensor_map(&mB1, a1->B, a1->K, a1->N, a1->ldb, 64))
      return false;
  } else {
    mA1 = mA0;
    mB1 = mB0;
  }
  atb_bf16_kernel<BN><<<unsigned(g0 + g1), kThreads, T::SMEM, s>>>(a0, a1 ? *a1 : a0, int(g0), int(mt0), int(mt1),
                                                                    mA0, mB0, mA1, mB1);
  return cudaGetLastError() == cudaSuccess;
}

}  // namespace

bool tn(const TnArgs& a0, int splits, bool bf16, cudaStream_t s) {
  if (a0.M <= 0 || a0.N <= 0 || a0.K < 0 || splits < 1) return a0.M <= 0 || a0.N <= 0;
  if (a0.k_per_split <= 0 || a0.k_per_split % kBK != 0) return false;
  // (cp.async of 16-byte chunks: bf16 rows must start 16-byte aligned)
  if (bf16 && ((reinterpret_cast<uintptr_t>(a0.A) & 15) || (reinterpret_cast<uintptr_t>(a0.B) & 15) ||
               (a0.lda * 2) % 16 || (a0.ldb * 2) % 16))
    return false;
  if (!bf16) {
    const long long mt = (a0.M + 63) / 64;
    const int nt = (a0.N + 63) / 64;
    if (mt > 0x7fffffff || splits > kMaxGridY || nt > kMaxGridY) return false;
    tn_f32_kernel<<<dim3(unsigned(mt), unsigned(splits), unsigned(nt)), 256, 0, s>>>(a0, 0);
    return cudaGetLastError() == cudaSuccess;
  }
  if (a0.epi == kEpiDsDq &&
      (a0.N > 256 || a0.N % 16 != 0 || !a0.nvalid || !a0.samp || !a0.S || !a0.dS || !a0.dqc || !a0.pooled ||
       a0.dim % 4 != 0 || a0.dim <= 0 || a0.N != 12 * a0.dim || a0.pooled_ld % 4 != 0 ||
       (reinterpret_cast<uintptr_t>(a0.S) & 15) || (reinterpret_cast<uintptr_t>(a0.dS) & 15) ||
       (reinterpret_cast<uintptr_t>(a0.dqc) & 15) || (reinterpret_cast<uintptr_t>(a0.pooled) & 15) ||
       a0.qoff[0] % 4 || a0.qoff[1] % 4 || a0.qoff[2] % 4))
    return false;
  if ((a0.epi == kEpiReluBias || a0.epi == kEpiMask) &&
      (a0.N > 256 || a0.N % 32 != 0 || !a0.H || a0.ldh % 8 || (reinterpret_cast<uintptr_t>(a0.H) & 15) ||
       (a0.HT && (a0.ldt % 8 || a0.ldt < (a0.M + 7) / 8 * 8 || (reinterpret_cast<uintptr_t>(a0.HT) & 15))) ||
       (a0.epi == kEpiMask && !a0.mask) || (a0.mask && a0.ldm < a0.N / 32) ||
       (a0.epi == kEpiReluBias && (!a0.bias || (reinterpret_cast<uintptr_t>(a0.bias) & 15)))))
    return false;
  // (the epilogue's fp32 stores are 16-byte vectors)
  if (a0.D && ((reinterpret_cast<uintptr_t>(a0.D) & 15) || a0.ldd % 4 || a0.split_stride % 4)) return false;
  // B resident (the products with a weight matrix as B): persistent CTAs
  if (splits == 1 && a0.K <= 4 * kBK && a0.N <= 256) {
    const int kb = int((a0.K + kBK - 1) / kBK);
    const int bn = a0.N <= 64 ? 64 : (a0.N <= 128 ? 128 : (a0.N <= 192 ? 192 : 256));
    int r = -1;
    if (bn == 64 && kb == 4) r = launch_resident<64, 4>(a0, s);
    else if (bn == 256 && kb == 3) r = launch_resident<256, 3>(a0, s);
    else if (bn == 256 && kb == 1) r = launch_resident<256, 1>(a0, s);
    else if (bn == 192 && kb == 4) r = launch_resident<192, 4>(a0, s);
    if (r >= 0) return r == 1;
  }
  // N in chunks of at most 256 columns: B's rows and D's columns move on
  for (int n0 = 0; n0 < a0.N; n0 += 256) {
    TnArgs a = a0;
    a.N = a0.N - n0 < 256 ? a0.N - n0 : 256;
    a.B = static_cast<const __nv_bfloat16*>(a0.B) + (long long)n0 * a0.ldb;
    a.D = a0.D + n0;
    bool ok;
    if (a.N <= 64) ok = launch_bf16<64>(a, splits, s);
    else if (a.N <= 128) ok = launch_bf16<128>(a, splits, s);
    else if (a.N <= 192) ok = launch_bf16<192>(a, splits, s);
    else ok = launch_bf16<256>(a, splits, s);
    if (!ok) return false;
  }
  return true;
}

namespace {
bool atb_ok(const TnArgs& a) {
  return a.k_per_split > 0 && a.k_per_split % kBK == 0 && a.D && !(reinterpret_cast<uintptr_t>(a.A) & 15) &&
         !(reinterpret_cast<uintptr_t>(a.B) & 15) && a.lda % 8 == 0 && a.ldb % 8 == 0 && a.lda >= a.M &&
         a.ldb >= a.N && !(reinterpret_cast<uintptr_t>(a.D) & 15) && a.ldd % 4 == 0 && a.split_stride % 4 == 0;
}
bool zero_splits(const TnArgs& a, int splits, cudaStream_t s) {
  for (int z = 0; z < splits; ++z)
    for (long long m = 0; m < a.M; ++m)
      if (cudaMemsetAsync(a.D + z * a.split_stride + m * a.ldd, 0, size_t(a.N) * 4, s) != cudaSuccess) return false;
  return true;
}
}  // namespace

bool atb(const TnArgs& a0, int splits, cudaStream_t s) {
  if (a0.M <= 0 || a0.N <= 0 || a0.K < 0 || splits < 1) return a0.M <= 0 || a0.N <= 0;
  if (!atb_ok(a0)) return false;
  if (a0.K == 0) return zero_splits(a0, splits, s);
  // N in chunks of at most 256 columns: B's columns and D's columns move on
  for (int n0 = 0; n0 < a0.N; n0 += 256) {
    TnArgs a = a0;
    a.N = a0.N - n0 < 256 ? a0.N - n0 : 256;
    a.B = static_cast<const __nv_bfloat16*>(a0.B) + n0;
    a.D = a0.D + n0;
    a.epi = kEpiF32;
    bool ok;
    if (a.N <= 64) ok = launch_atb<64>(a, splits, nullptr, 0, s);
    else if (a.N <= 128) ok = launch_atb<128>(a, splits, nullptr, 0, s);
    else if (a.N <= 192) ok = launch_atb<192>(a, splits, nullptr, 0, s);
    else ok = launch_atb<256>(a, splits, nullptr, 0, s);
    if (!ok) return false;
  }
  return true;
}

bool atb2(const TnArgs& a0, int s0, const TnArgs& a1, int s1, cudaStream_t s) {
  const bool e0 = a0.M <= 0 || a0.N <= 0, e1 = a1.M <= 0 || a1.N <= 0;
  if (e0 || e1 || a0.N > 256 || a1.N > 256 || a0.K <= 0 || a1.K <= 0)
    return atb(a0, s0, s) && atb(a1, s1, s);
  if (s0 < 1 || s1 < 1 || !atb_ok(a0) || !atb_ok(a1)) return false;
  TnArgs b0 = a0, b1 = a1;
  b0.epi = b1.epi = kEpiF32;
  return launch_atb<256>(b0, s0, &b1, s1, s);
}

bool reduce(const float* P, long long split_stride, int splits, long long ldp, float* D, long long ldd, long long M,
            int N, cudaStream_t s) {
  return reduce2(P, split_stride, splits, ldp, D, ldd, M, N, nullptr, 0, 0, 0, nullptr, 0, 0, 0, s);
}

bool reduce2(const float* P0, long long ss0, int splits0, long long ldp0, float* D0, long long ldd0, long long M0,
             int N0, const float* P1, long long ss1, int splits1, long long ldp1, float* D1, long long ldd1,
             long long M1, int N1, cudaStream_t s) {
  const long long t0 = M0 * N0, t1 = P1 ? M1 * N1 : 0;
  if (t0 <= 0 && t1 <= 0) return true;
  // blocks in proportion to the outputs, about 8 per SM in all
  auto blocks = [](long long t) { return t <= 0 ? 0LL : ((t + 31) / 32 < 152 * 8 ? (t + 31) / 32 : 152LL * 8); };
  long long b0 = blocks(t0), b1 = blocks(t1);
  if (b0 + b1 > 152 * 8 && t0 > 0 && t1 > 0) {
    b0 = 152 * 8 * t0 / (t0 + t1);
    b0 = b0 < 1 ? 1 : b0;
    b1 = 152 * 8 - b0;
    b1 = b1 < 1 ? 1 : b1;
  }
  const RedJob j0{P0, ss0, ldp0, ldd0, t0 > 0 ? M0 : 0, D0, splits0, N0 > 0 ? N0 : 1};
  const RedJob j1{P1, ss1, ldp1, ldd1, t1 > 0 ? M1 : 0, D1, splits1, N1 > 0 ? N1 : 1};
  auto vec = [](const RedJob& j) {
    return j.M == 0 || (j.N % 4 == 0 && j.ldp % 4 == 0 && j.ldd % 4 == 0 && j.split_stride % 4 == 0 &&
                        !(reinterpret_cast<uintptr_t>(j.P) & 15) && !(reinterpret_cast<uintptr_t>(j.D) & 15));
  };
  if (vec(j0) && vec(j1)) {
    auto blocks4 = [](long long t) { return t <= 0 ? 0LL : ((t / 4 + 31) / 32 < 152 * 4 ? (t / 4 + 31) / 32 : 152LL * 4); };
    long long c0 = blocks4(t0), c1 = blocks4(t1);
    reduce4_kernel<<<unsigned(c0 + c1), 256, 0, s>>>(j0, j1, int(c0));
  } else {
    reduce_kernel<<<unsigned(b0 + b1), 256, 0, s>>>(j0, j1, int(b0));
  }
  return cudaGetLastError() == cudaSuccess;
}

bool transpose(const void* in, long long ld_in, long long rows, int cols, void* out, long long ld_out, int esize,
               cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return true;
  const long long gx = (rows + 31) / 32;
  const int gy = (cols + 31) / 32;
  if (gx > 0x7fffffff || gy > kMaxGridY) return false;
  const dim3 grid{static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1u};
  const dim3 block{32u, 8u, 1u};
  if (esize == 2 && ld_in % 8 == 0 && ld_out % 8 == 0 && (reinterpret_cast<uintptr_t>(in) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    const long long hx = (rows + 63) / 64;
    const int hy = (cols + 63) / 64;
    if (hx > 0x7fffffff || hy > kMaxGridY) return false;
    transpose16_kernel<<<dim3{static_cast<unsigned>(hx), static_cast<unsigned>(hy), 1u}, 256, 0, s>>>(
        static_cast<const uint16_t*>(in), ld_in, rows, cols, static_cast<uint16_t*>(out), ld_out);
  } else if (esize == 2)
    transpose_kernel<uint16_t><<<grid, block, 0, s>>>(static_cast<const uint16_t*>(in), ld_in, rows, cols,
                                                       static_cast<uint16_t*>(out), ld_out);
  else if (esize == 4)
    transpose_kernel<uint32_t><<<grid, block, 0, s>>>(static_cast<const uint32_t*>(in), ld_in, rows, cols,
                                                       static_cast<uint32_t*>(out), ld_out);
  else
    return false;
  return cudaGetLastError() == cudaSuccess;
}

}  // namespace gemm
}  // namespace dsf
