// The dense towers after the sparse path (MultiTowerDIN: current state
// analysis, section 4.4; model config, section 7): the deep tower
// pooled[256] -> 512 -> 256 -> 128 and the final tower cat[deep, din] (176) ->
// 64 -> 1 (the logit), ReLU after every hidden layer.
//
// One CTA of 512 threads takes 128 samples. Every layer is a bf16 tcgen05 MMA
// (M = 128 samples, fp32 accumulators in tensor memory) with both operands in
// shared memory, K-major and 128-byte swizzled: the activations are written
// there by the epilogue of the previous layer (bias, ReLU, bf16), the weights
// arrive by bulk copy in 64-wide K-blocks -- through a two-stage ring for the
// two 256 KB layers, whole for the last two. Shared memory holds three 64 KB
// regions X0 X1 X2 whose roles change per layer:
//   layer 1: A = pooled (X0), W1 K-blocks (64 KB) in X1 / X2
//   layer 2: A = h1 (X0 X1), W2 K-blocks (32 KB) in the two halves of X2
//   layer 3: A = h2 (X1), W3 (64 KB) in X0
//   layer 4: A = cat[h3, din, 0] (X1), Wf (24 KB) in X2
// Thread 0 issues the copies and the MMAs; every wait is bounded and a
// timeout sets DSF_FLAG_TIMEOUT instead of hanging.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <type_traits>

#include "dinsparse.h"
#include "ptx.cuh"

namespace dsf {
namespace towers {

constexpr int kP = 256, kH1 = 512, kH2 = 256, kH3 = 128, kDQ = 48, kKF = 176, kKFP = 192, kHF = 64;
constexpr int kTM = 128, kThreads = 512, kWarps = kThreads / 32;
constexpr int kBlk = 64;  // K elements per K-block (128 bytes of bf16)

// packed bf16 weights in the workspace: K-blocks of [N rows x 128 B]
constexpr size_t kW1Off = 0, kW1B = size_t(kH1) * kP * 2;
constexpr size_t kW2Off = kW1Off + kW1B, kW2B = size_t(kH2) * kH1 * 2;
constexpr size_t kW3Off = kW2Off + kW2B, kW3B = size_t(kH3) * kH2 * 2;
constexpr size_t kWfOff = kW3Off + kW3B, kWfB = size_t(kHF) * kKFP * 2;
constexpr size_t kWsTag = kWfOff + kWfB;  // prepared tag
constexpr size_t kWsBytes = kWsTag + 256;
constexpr uint32_t kTowersTag = 0x544f5752u;  // 'TOWR'

constexpr int kXB = 64 * 1024;                 // one region
constexpr int kX0 = 0, kX1 = kXB, kX2 = 2 * kXB;
constexpr int kAB = kTM * 128;                 // one 64-wide K-block of an activation (16 KB)

struct Misc {
  float bd1[kH1], bd2[kH2], bd3[kH3], bf1[kHF], wo[kHF];
  float red[4][kTM];
  uint64_t full[2], done[2], mma, w3, wf;
  uint32_t tmem_base;
  int abort_;
};
constexpr int kMiscOff = 3 * kXB;
constexpr int kSmem = kMiscOff + int(sizeof(Misc)) + 1024;
static_assert(kSmem <= 227 * 1024, "towers: shared memory per block");

struct Params {
  const float* pooled;  // [B, 256]
  const float* din;     // [B, 48]
  const float *bd1, *bd2, *bd3, *bf1, *wo, *bo;
  const uint8_t* wpack;
  const uint32_t* tag;
  float* logit;  // [B]
  int B;
  int* status;
};

// Element (row, k) of a K-major, 128-byte-swizzled bf16 operand of `rows`
// rows made of 64-wide K-blocks.
__device__ __forceinline__ uint32_t xoff(int row, int k, int rows) {
  return sw128_offset(uint32_t(row), uint32_t(k), uint32_t(rows));
}

__global__ void __launch_bounds__(kThreads, 1) towers_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc* ms = reinterpret_cast<Misc*>(sm + kMiscOff);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s0 = blockIdx.x * kTM;
  const int n = min(kTM, p.B - s0);
  int local_flags = 0;
  const bool prepared = *p.tag == kTowersTag;

  // ---------------------------------------------------------------- prologue
  auto load = [&](uint8_t* dst, size_t src_off, uint32_t bytes, uint64_t* bar) {  // thread 0
    mbar_arrive_expect_tx(bar, bytes);
    for (uint32_t o = 0; o < bytes; o += 16384)
      bulk_g2s(dst + o, p.wpack + src_off + o, min(16384u, bytes - o), bar);
  };
  if (tid == 0) {
    ms->abort_ = prepared ? 0 : 1;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->full[i], 1);
      mbar_init(&ms->done[i], 1);
    }
    mbar_init(&ms->mma, 1);
    mbar_init(&ms->w3, 1);
    mbar_init(&ms->wf, 1);
    fence_mbarrier_init();
    if (prepared) {  // W1 K-blocks 0 and 1
      load(sm + kX1, kW1Off, kH1 * 128, &ms->full[0]);
      load(sm + kX2, kW1Off + size_t(kH1) * 128, kH1 * 128, &ms->full[1]);
    }
  }
  if (warp == 0) {
    __syncwarp();  // the allocation is warp-collective: converge after thread 0's branch
    tmem_alloc(&ms->tmem_base, 512);
    tmem_relinquish();
    tc_fence_before();
  }
  for (int i = tid; i < kH1; i += kThreads) ms->bd1[i] = p.bd1[i];
  for (int i = tid; i < kH2; i += kThreads) ms->bd2[i] = p.bd2[i];
  if (tid < kH3) ms->bd3[tid] = p.bd3[tid];
  if (tid < kHF) {
    ms->bf1[tid] = p.bf1[tid];
    ms->wo[tid] = p.wo[tid];
  }
  // layer-1 A: the pooled rows as bf16, 8 elements (one 16-byte chunk) per
  // item; a thread's items are loaded in batches of kPB before any is stored,
  // so each thread keeps kPB * 32 bytes in flight instead of one round trip
  // per item
  {
    constexpr int kItems = kTM * (kP / 8) / kThreads, kPB = 8;
    static_assert(kItems % kPB == 0, "towers: pooled batches");
#pragma unroll 1
    for (int i0 = 0; i0 < kItems; i0 += kPB) {
      float4 a[kPB], b[kPB];
#pragma unroll
      for (int j = 0; j < kPB; ++j) {
        const int c = tid + (i0 + j) * kThreads, r = c / (kP / 8), k = (c - r * (kP / 8)) * 8;
        const float4* src = reinterpret_cast<const float4*>(p.pooled + (long long)(s0 + r) * kP + k);
        a[j] = r < n ? __ldg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
        b[j] = r < n ? __ldg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kPB; ++j) {
        const int c = tid + (i0 + j) * kThreads, r = c / (kP / 8), k = (c - r * (kP / 8)) * 8;
        *reinterpret_cast<uint4*>(sm + kX0 + xoff(r, k, kTM)) =
            make_uint4(pack_bf16x2(a[j].x, a[j].y), pack_bf16x2(a[j].z, a[j].w), pack_bf16x2(b[j].x, b[j].y),
                       pack_bf16x2(b[j].z, b[j].w));
      }
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ms->tmem_base;
  const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
  const int row = (warp & 3) * 32 + lane;  // this thread's accumulator row

  uint32_t gblk = 0;       // streamed K-blocks so far (ring stage gblk & 1)
  uint32_t mma_phase = 0;  // completions of ms->mma so far
  // thread 0: one layer's MMAs over nkb K-blocks. a(kb): A descriptor base of
  // K-block kb; b(kb, st): B base (stage st when streamed); nh N-halves of 256.
  auto fail = [&]() { ms->abort_ = 2; };
  constexpr uint32_t ID256 = idesc_bf16_f32(kTM, 256), ID128 = idesc_bf16_f32(kTM, 128),
                     ID64 = idesc_bf16_f32(kTM, 64);
  // streamed layer: weights of nkb K-blocks of `blk` bytes from src_off, two
  // blocks already on their way (gblk, gblk + 1)
  auto stream_layer = [&](uint32_t a_base, int nkb, size_t src_off, uint32_t blk, uint8_t* stage0,
                          uint8_t* stage1, int nh, uint32_t idesc) {
    for (int kb = 0; kb < nkb && ms->abort_ == 0; ++kb, ++gblk) {
      const uint32_t st = gblk & 1u, ph = (gblk >> 1) & 1u;
      if (!mbar_wait(&ms->full[st], ph)) { fail(); break; }
      tc_fence_after();
      const uint32_t wb = smem_u32(st ? stage1 : stage0);
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk)
        for (int h = 0; h < nh; ++h)
          tc_mma_f16(tbase + uint32_t(h * 256), sw128_kmajor_desc(a_base + kb * kAB + kk * 32),
                     sw128_kmajor_desc(wb + h * 256 * 128 + kk * 32), idesc, (kb | kk) ? 1u : 0u);
      tc_commit(&ms->done[st]);
      // the previous block's MMAs done: its stage takes block kb + 1
      if (kb >= 1 && kb + 1 < nkb) {
        const uint32_t pst = (gblk - 1u) & 1u, pph = ((gblk - 1u) >> 1) & 1u;
        if (!mbar_wait(&ms->done[pst], pph)) { fail(); break; }
        load(pst ? stage1 : stage0, src_off + size_t(kb + 1) * blk, blk, &ms->full[pst]);
      }
    }
    // the last block's commit covers every MMA of the layer
    if (ms->abort_ == 0 && !mbar_wait(&ms->done[(gblk - 1u) & 1u], ((gblk - 1u) >> 1) & 1u)) fail();
  };
  // resident layer: all nkb K-blocks in smem at w_base
  auto resident_layer = [&](uint32_t a_base, int nkb, uint32_t w_base, uint32_t wblk, uint32_t idesc) {
#pragma unroll 1
    for (int kb = 0; kb < nkb; ++kb)
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk)
        tc_mma_f16(tbase, sw128_kmajor_desc(a_base + kb * kAB + kk * 32),
                   sw128_kmajor_desc(w_base + kb * wblk + kk * 32), idesc, (kb | kk) ? 1u : 0u);
    tc_commit(&ms->mma);
  };
  auto wait_mma = [&]() {  // thread 0
    if (!mbar_wait(&ms->mma, mma_phase & 1u)) fail();
    ++mma_phase;
  };
  // epilogue: accumulator columns [c0, c0 + 16 NB) of this thread's row ->
  // ReLU(acc + bias) as bf16 into the next layer's A operand at K offset c0.
  // The NB loads are issued before one wait: the wait covers every load in
  // flight, so batching pays its latency once per 16 NB columns.
  auto epi_store = [&](auto nb_tag, int c0, const float* bias, uint8_t* dst) {
    constexpr int NB = decltype(nb_tag)::value;
    float v[16 * NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) tmem_ld16(tbase + lane_base + uint32_t(c0 + 16 * b), v + 16 * b);
    tmem_ld_wait();
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const int c = c0 + 16 * b;
      uint32_t h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        h[e] = pack_bf16x2_relu(v[16 * b + 2 * e] + bias[c + 2 * e], v[16 * b + 2 * e + 1] + bias[c + 2 * e + 1]);
      *reinterpret_cast<uint4*>(dst + xoff(row, c, kTM)) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(dst + xoff(row, c + 8, kTM)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
  };
  // all warps: wait for the layer's MMAs (thread 0 waited already), then read
  auto sync_after_mma = [&]() {
    __syncthreads();
    tc_fence_after();
  };
  auto sync_before_mma = [&]() {  // smem operands written, accumulator reads done
    tmem_ld_wait();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
  };

  // ---------------------------------------------------------------- layer 1
  if (tid == 0 && ms->abort_ == 0) {
    stream_layer(smem_u32(sm + kX0), kP / kBlk, kW1Off, kH1 * 128, sm + kX1, sm + kX2, 2, ID256);
    // W2 blocks 0 and 1 into the two halves of X2 (W1 is done with it)
    if (ms->abort_ == 0) {
      load(sm + kX2 + (gblk & 1u) * (kXB / 2), kW2Off, kH2 * 128, &ms->full[gblk & 1u]);
      load(sm + kX2 + ((gblk + 1u) & 1u) * (kXB / 2), kW2Off + size_t(kH2) * 128, kH2 * 128,
           &ms->full[(gblk + 1u) & 1u]);
    }
  }
  sync_after_mma();
  if (ms->abort_ == 0) {
    // h1 [128 x 512] -> X0 X1 (8 K-blocks); warp w: columns 128 (w / 4) .. + 128
#pragma unroll 1
    for (int c = (warp >> 2) * 128; c < (warp >> 2) * 128 + 128; c += 64)
      epi_store(std::integral_constant<int, 4>{}, c, ms->bd1, sm + kX0);
  }
  sync_before_mma();

  // ---------------------------------------------------------------- layer 2
  if (tid == 0 && ms->abort_ == 0) {
    tc_fence_after();
    // the stages alternate with gblk: stage s sits in half s of X2
    stream_layer(smem_u32(sm + kX0), kH1 / kBlk, kW2Off, kH2 * 128, sm + kX2, sm + kX2 + kXB / 2, 1, ID256);
    if (ms->abort_ == 0) {  // W3 into X0 and Wf into X2, both free once layer 2 is done
      load(sm + kX0, kW3Off, uint32_t(kW3B), &ms->w3);
      load(sm + kX2, kWfOff, uint32_t(kWfB), &ms->wf);
    }
  }
  sync_after_mma();
  if (ms->abort_ == 0) {
    // h2 [128 x 256] -> X1 (4 K-blocks); warp w: columns 64 (w / 4) .. + 64
    epi_store(std::integral_constant<int, 4>{}, (warp >> 2) * 64, ms->bd2, sm + kX1);
  }
  sync_before_mma();

  // ---------------------------------------------------------------- layer 3
  if (tid == 0 && ms->abort_ == 0) {
    tc_fence_after();
    if (!mbar_wait(&ms->w3, 0)) fail();
    else {
      tc_fence_after();
      resident_layer(smem_u32(sm + kX1), kH2 / kBlk, smem_u32(sm + kX0), kH3 * 128, ID128);
      wait_mma();
    }
  }
  sync_after_mma();
  if (ms->abort_ == 0) {
    // cat[h3, din, 0] [128 x 192] -> X1 (3 K-blocks): h3 in K 0..127, warp w:
    // columns 32 (w / 4) .. + 32 ...
    epi_store(std::integral_constant<int, 2>{}, (warp >> 2) * 32, ms->bd3, sm + kX1);
  }
  // ... and din (fp32 -> bf16) in K 128..175, zeros in K 176..191
  {
    constexpr int kItems = kTM * (kKFP - kH3) / 8 / kThreads;
    float4 a[kItems], b[kItems];
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
      const int c = tid + j * kThreads, r = c / ((kKFP - kH3) / 8), k = kH3 + (c - r * ((kKFP - kH3) / 8)) * 8;
      const float4* src = reinterpret_cast<const float4*>(p.din + (long long)(s0 + r) * kDQ + (k - kH3));
      const bool in = r < n && k < kKF;
      a[j] = in ? __ldg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
      b[j] = in ? __ldg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
      const int c = tid + j * kThreads, r = c / ((kKFP - kH3) / 8), k = kH3 + (c - r * ((kKFP - kH3) / 8)) * 8;
      *reinterpret_cast<uint4*>(sm + kX1 + xoff(r, k, kTM)) =
          make_uint4(pack_bf16x2(a[j].x, a[j].y), pack_bf16x2(a[j].z, a[j].w), pack_bf16x2(b[j].x, b[j].y),
                     pack_bf16x2(b[j].z, b[j].w));
    }
  }
  sync_before_mma();

  // ---------------------------------------------------------------- layer 4
  if (tid == 0 && ms->abort_ == 0) {
    tc_fence_after();
    if (!mbar_wait(&ms->wf, 0)) fail();
    else {
      tc_fence_after();
      resident_layer(smem_u32(sm + kX1), kKFP / kBlk, smem_u32(sm + kX2), kHF * 128, ID64);
      wait_mma();
    }
  }
  sync_after_mma();
  // the logit: w_o . ReLU(acc + b_f1) + b_o; warp w sums columns 16 (w / 4) .. + 16
  if (ms->abort_ == 0) {
    const int cg = warp >> 2;
    float v[16];
    tmem_ld16(tbase + lane_base + uint32_t(cg * 16), v);
    tmem_ld_wait();
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) part = fmaf(fmaxf(v[e] + ms->bf1[cg * 16 + e], 0.f), ms->wo[cg * 16 + e], part);
    ms->red[cg][row] = part;
  }
  tc_fence_before();
  __syncthreads();
  if (ms->abort_ == 0 && tid < n)
    p.logit[s0 + tid] = ((ms->red[0][tid] + ms->red[1][tid]) + (ms->red[2][tid] + ms->red[3][tid])) + __ldg(p.bo);

  // ---------------------------------------------------------------- cleanup
  if (tid == 0) {
    const int a = ms->abort_;
    if (a == 1) local_flags |= DSF_FLAG_NOT_PREPARED;
    if (a == 2) {
      local_flags |= DSF_FLAG_TIMEOUT;
      // give copies and MMAs in flight one more bounded wait before TMEM and
      // shared memory are released
      mbar_wait(&ms->mma, mma_phase & 1u);
      for (int i = 0; i < 2; ++i) mbar_wait(&ms->done[i], 0), mbar_wait(&ms->full[i], 0);
      mbar_wait(&ms->w3, 0);
      mbar_wait(&ms->wf, 0);
    }
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (tid == 0 && local_flags && p.status) atomicOr(p.status, local_flags);
}

// Packs the fp32 [out, in] tower weights into bf16 K-major 128-byte-swizzled
// K-blocks (Wf padded to K = 192 with zeros) and writes the prepared tag last.
__global__ void prepare_towers_kernel(const float* __restrict__ Wd1, const float* __restrict__ Wd2,
                                      const float* __restrict__ Wd3, const float* __restrict__ Wf1,
                                      uint8_t* ws) {
  const long long n1 = (long long)kH1 * kP, n2 = (long long)kH2 * kH1, n3 = (long long)kH3 * kH2,
                  n4 = (long long)kHF * kKFP;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n1 + n2 + n3 + n4;
       i += (long long)gridDim.x * blockDim.x) {
    float w;
    size_t off;
    if (i < n1) {
      const int r = int(i / kP), k = int(i % kP);
      w = Wd1[i];
      off = kW1Off + sw128_offset(r, k, kH1);
    } else if (i < n1 + n2) {
      const long long j = i - n1;
      const int r = int(j / kH1), k = int(j % kH1);
      w = Wd2[j];
      off = kW2Off + sw128_offset(r, k, kH2);
    } else if (i < n1 + n2 + n3) {
      const long long j = i - n1 - n2;
      const int r = int(j / kH2), k = int(j % kH2);
      w = Wd3[j];
      off = kW3Off + sw128_offset(r, k, kH3);
    } else {
      const long long j = i - n1 - n2 - n3;
      const int r = int(j / kKFP), k = int(j % kKFP);
      w = k < kKF ? Wf1[(long long)r * kKF + k] : 0.f;
      off = kWfOff + sw128_offset(r, k, kHF);
    }
    *reinterpret_cast<__nv_bfloat16*>(ws + off) = __float2bfloat16_rn(w);
  }
}

__global__ void towers_tag_kernel(uint32_t* tag) { *tag = kTowersTag; }

bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

}  // namespace towers
}  // namespace dsf

using namespace dsf::towers;

extern "C" size_t dsf_towers_workspace_bytes(void) { return kWsBytes; }

extern "C" int dsf_prepare_towers(const dsf_towers* t, void* ws, size_t ws_bytes, void* stream) {
  if (!t || !t->Wd1 || !t->Wd2 || !t->Wd3 || !t->Wf1) return DSF_EINVAL;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < kWsBytes) return DSF_EWORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  prepare_towers_kernel<<<256, 256, 0, s>>>(t->Wd1, t->Wd2, t->Wd3, t->Wf1, w);
  if (cudaGetLastError() != cudaSuccess) return DSF_ECUDA;
  towers_tag_kernel<<<1, 1, 0, s>>>(reinterpret_cast<uint32_t*>(w + kWsTag));
  return cudaGetLastError() == cudaSuccess ? DSF_OK : DSF_ECUDA;
}

extern "C" int ctr_towers_fwd(const float* pooled_dev, const float* din_dev, int32_t B, const dsf_towers* t,
                              float* logit_dev, const void* ws, size_t ws_bytes, int32_t* status_dev,
                              void* stream) {
  if (B < 0 || !t) return DSF_EINVAL;
  if (B == 0) return DSF_OK;
  if (!pooled_dev || !din_dev || !logit_dev || !aligned16(pooled_dev) || !aligned16(din_dev)) return DSF_EINVAL;
  if (!t->bd1 || !t->bd2 || !t->bd3 || !t->bf1 || !t->wo || !t->bo) return DSF_EINVAL;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < kWsBytes) return DSF_EWORKSPACE;
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSF_ECUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(towers_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
      return DSF_EUNSUPPORTED;
    attr_set[dev] = true;
  }
  Params p{};
  p.pooled = pooled_dev;
  p.din = din_dev;
  p.bd1 = t->bd1;
  p.bd2 = t->bd2;
  p.bd3 = t->bd3;
  p.bf1 = t->bf1;
  p.wo = t->wo;
  p.bo = t->bo;
  p.wpack = static_cast<const uint8_t*>(ws);
  p.tag = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(ws) + kWsTag);
  p.logit = logit_dev;
  p.B = B;
  p.status = status_dev;
  const int grid = (B + kTM - 1) / kTM;
  towers_kernel<<<grid, kThreads, kSmem, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? DSF_OK : DSF_ECUDA;
}
