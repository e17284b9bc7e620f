// C ABI of the sparse forward (declared in include/dinsparse.h): argument
// validation, workspace layout, MLP weight packing and kernel dispatch. No
// function here allocates device memory; every buffer belongs to the caller.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "dinsparse.h"
#include "abi_checks.cuh"
#include "launch.cuh"

namespace dsf {
namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t wpack, w1t, w2t, qbuf, total;
};

WsLayout ws_layout(int32_t B, int32_t D) {
  WsLayout l{};
  const size_t K1 = size_t(12) * D;
  l.wpack = kWsWpackOff;
  l.w1t = align256(l.wpack + (size_t(kN1) * K1 + size_t(kN2) * kN1) * 2);
  l.w2t = align256(l.w1t + K1 * kN1 * 4);
  l.qbuf = align256(l.w2t + size_t(kN1) * kN2 * 4);
  l.total = align256(l.qbuf + size_t(B > 0 ? B : 0) * 3 * D * 4);
  return l;
}


// Packs W1 / W2 (fp32, [out, in]) into bf16 K-major 128-byte-swizzled operand
// blocks and fp32 transposed copies; writes the prepared tag last.
__global__ void prepare_kernel(const float* __restrict__ W1, const float* __restrict__ W2, int K1,
                               uint8_t* wpack, float* w1t, float* w2t) {
  const long long n1 = (long long)kN1 * K1, n2 = (long long)kN2 * kN1;
  const long long W1B = n1 * 2;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n1 + n2;
       i += (long long)gridDim.x * blockDim.x) {
    if (i < n1) {
      const int n = int(i / K1), k = int(i % K1);
      const float w = W1[i];
      *reinterpret_cast<__nv_bfloat16*>(wpack + sw128_offset(n, k, kN1)) = __float2bfloat16_rn(w);
      w1t[(long long)k * kN1 + n] = w;
    } else {
      const long long j = i - n1;
      const int n = int(j / kN1), k = int(j % kN1);
      const float w = W2[j];
      *reinterpret_cast<__nv_bfloat16*>(wpack + W1B + sw128_offset(n, k, kN2)) = __float2bfloat16_rn(w);
      w2t[(long long)k * kN2 + n] = w;
    }
  }
}

__global__ void tag_kernel(uint32_t* magic, uint32_t tag) { *magic = tag; }

int check_ws(void* ws, size_t bytes, int32_t B, int32_t D) {
  if (!ws || !aligned(ws, 256)) return DSF_EWORKSPACE;
  if (bytes < ws_layout(B, D).total) return DSF_EWORKSPACE;
  return DSF_OK;
}

void fill_common(FwdParams& p, const dsf_tables* t, const dsf_kjt* k, int32_t B, void* ws,
                 int32_t* status) {
  std::memset(&p, 0, sizeof(p));
  hash::Layout L{};
  uint8_t* hw = nullptr;
  if (t->hash) {
    L = hash::layout(t->hash->capacity, t->hash->D, t->dtype == DSF_BF16 ? 2 : 4);
    hw = static_cast<uint8_t*>(t->hash->workspace);
    p.hkeys = reinterpret_cast<const unsigned long long*>(hw + L.keys_off);
    p.hhdr = reinterpret_cast<const hash::Header*>(hw);
    p.hbmask = L.n_buckets - 1;
    p.hslots = L.n_slots;
  }
  for (int f = 0; f < t->F; ++f) {
    if (hashed(t, f)) {  // the fused row pool; the zero row is the last
      p.tables[f] = hw + L.pool_off;
      p.rows[f] = static_cast<long long>(L.n_slots) + 1;
      p.hash_mask |= 1u << f;
      p.kspace[f] = static_cast<unsigned char>(t->hash->key_space[f]);
    } else {
      p.tables[f] = t->table_ptrs[f];
      p.rows[f] = t->table_rows[f];
    }
    if (t->pooling && t->pooling[f] == DSF_POOL_MEAN) p.mean_mask |= 1u << f;
  }
  p.F = t->F;
  p.B = B;
  p.values = reinterpret_cast<const long long*>(k->values_dev);
  p.n_values = k->n_values;
  p.lengths = k->lengths_dev;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.magic = reinterpret_cast<const uint32_t*>(w + kWsMagicOff);
  p.epoch = reinterpret_cast<unsigned int*>(w + kWsEpochOff);
  p.partials = reinterpret_cast<unsigned long long*>(w + kWsPartOff);
  p.status = status;
}

int map_launch(int rc) {
  if (rc == 0) return DSF_OK;
  if (rc == 2) return DSF_EUNSUPPORTED;
  return DSF_ECUDA;
}

int run_attention(const dsf_tables* tables, const dsf_kjt* kjt, const dsf_seq* seq,
                  const int32_t q_feat[3], const int32_t seq_table[3], int32_t B,
                  const dsf_mlp* mlp, float* pooled, float* din, float* logits, void* ws,
                  size_t ws_bytes, int32_t* status, void* stream) {
  int rc;
  if ((rc = check_tables(tables)) != DSF_OK) return rc;
  if (B < 0 || B > (1 << 24)) return DSF_EINVAL;
  if ((rc = check_kjt(kjt, B, tables->F)) != DSF_OK) return rc;
  if ((rc = check_seq(seq, B)) != DSF_OK) return rc;
  if ((rc = check_mlp(mlp, tables->D)) != DSF_OK) return rc;
  // the tensor-core MLP with D = 64 is built for bf16 tables only
  if (mlp->mode == DSF_MODE_BF16_TC && tables->D == 64 && tables->dtype != DSF_BF16) return DSF_EUNSUPPORTED;
  if (!q_feat || !seq_table) return DSF_EINVAL;
  for (int k = 0; k < 3; ++k) {
    if (q_feat[k] < 0 || q_feat[k] >= tables->F) return DSF_EINVAL;
    if (seq_table[k] < 0 || seq_table[k] >= tables->F) return DSF_EINVAL;
  }
  if (!din || !aligned(din, 16)) return DSF_EINVAL;
  if (pooled && !aligned(pooled, 16)) return DSF_EINVAL;
  if (logits && !aligned(logits, 4)) return DSF_EINVAL;
  if ((rc = check_ws(ws, ws_bytes, B, tables->D)) != DSF_OK) return rc;
  if (B == 0) return DSF_OK;
  const WsLayout l = ws_layout(B, tables->D);
  FwdParams p;
  fill_common(p, tables, kjt, B, ws, status);
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.max_len = seq->max_len;
  p.seq_values = reinterpret_cast<const long long*>(seq->values_dev);
  p.n_seq = seq->n_per_key;
  p.seq_lengths = seq->lengths_dev;
  for (int k = 0; k < 3; ++k) {
    p.q_feat[k] = q_feat[k];
    p.seq_table[k] = seq_table[k];
  }
  p.pooled = pooled;
  p.qbuf = reinterpret_cast<float*>(w + l.qbuf);
  p.din = din;
  p.logits = logits;
  p.b1 = mlp->b1;
  p.b2 = mlp->b2;
  p.w3 = mlp->w3;
  p.b3 = mlp->b3;
  p.wpack = w + l.wpack;
  p.w1t = reinterpret_cast<const float*>(w + l.w1t);
  p.w2t = reinterpret_cast<const float*>(w + l.w2t);
  const bool bf16 = tables->dtype == DSF_BF16;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int lrc = mlp->mode == DSF_MODE_BF16_TC ? launch_attn_tc(tables->D, bf16, p, s)
                                                 : launch_attn_f32(tables->D, bf16, p, s);
  return map_launch(lrc);
}

}  // namespace
}  // namespace dsf

using namespace dsf;

extern "C" {

size_t dsf_workspace_bytes(int32_t B, int32_t D) {
  if (D != 16 && D != 64) return 0;
  return ws_layout(B, D).total;
}

int dsf_workspace_init(void* workspace_dev, size_t ws_bytes, void* stream) {
  if (!workspace_dev || !aligned(workspace_dev, 256) || ws_bytes < kWsWpackOff) return DSF_EWORKSPACE;
  const cudaError_t e = cudaMemsetAsync(workspace_dev, 0, kWsWpackOff, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSF_OK : DSF_ECUDA;
}

int dsf_prepare_mlp(const dsf_mlp* mlp, int32_t D, void* workspace_dev, size_t ws_bytes, void* stream) {
  if (D != 16 && D != 64) return DSF_EUNSUPPORTED;
  if (!mlp || !mlp->W1 || !mlp->W2) return DSF_EINVAL;
  if (mlp->K1 != 12 * D || mlp->N1 != kN1 || mlp->N2 != kN2) return DSF_EUNSUPPORTED;
  if (!workspace_dev || !aligned(workspace_dev, 256) || ws_bytes < ws_layout(0, D).total)
    return DSF_EWORKSPACE;
  const WsLayout l = ws_layout(0, D);
  uint8_t* w = static_cast<uint8_t*>(workspace_dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long n = (long long)kN1 * 12 * D + (long long)kN2 * kN1;
  const int threads = 256;
  const int blocks = int((n + threads - 1) / threads);
  prepare_kernel<<<blocks, threads, 0, s>>>(mlp->W1, mlp->W2, 12 * D, w + l.wpack,
                                            reinterpret_cast<float*>(w + l.w1t),
                                            reinterpret_cast<float*>(w + l.w2t));
  tag_kernel<<<1, 1, 0, s>>>(reinterpret_cast<uint32_t*>(w + kWsMagicOff), kMagicBase | uint32_t(D));
  return cudaGetLastError() == cudaSuccess ? DSF_OK : DSF_ECUDA;
}

int emb_bag_pool(const dsf_tables* tables, const dsf_kjt* kjt, int32_t B, float* pooled_dev,
                 void* workspace_dev, size_t ws_bytes, int32_t* status_dev, void* stream) {
  int rc;
  if ((rc = check_tables(tables)) != DSF_OK) return rc;
  if (B < 0 || B > (1 << 24)) return DSF_EINVAL;
  if ((rc = check_kjt(kjt, B, tables->F)) != DSF_OK) return rc;
  if (!pooled_dev || !aligned(pooled_dev, 16)) return DSF_EINVAL;
  if ((rc = check_ws(workspace_dev, ws_bytes, B, tables->D)) != DSF_OK) return rc;
  if (B == 0) return DSF_OK;
  FwdParams p;
  fill_common(p, tables, kjt, B, workspace_dev, status_dev);
  p.pooled = pooled_dev;
  p.max_len = 1;
  return map_launch(launch_pool(tables->D, tables->dtype == DSF_BF16, p,
                                static_cast<cudaStream_t>(stream)));
}

int din_jagged_attn(const dsf_tables* tables, const dsf_kjt* kjt, const dsf_seq* seq,
                    const int32_t q_feat[3], const int32_t seq_table[3], int32_t B,
                    const dsf_mlp* mlp, float* din_dev, float* logits_dev, void* workspace_dev,
                    size_t ws_bytes, int32_t* status_dev, void* stream) {
  return run_attention(tables, kjt, seq, q_feat, seq_table, B, mlp, nullptr, din_dev, logits_dev,
                       workspace_dev, ws_bytes, status_dev, stream);
}

int din_sparse_fwd(const dsf_tables* tables, const dsf_kjt* kjt, const dsf_seq* seq,
                   const int32_t q_feat[3], const int32_t seq_table[3], int32_t B,
                   const dsf_mlp* mlp, float* pooled_dev, float* din_dev, float* logits_dev,
                   void* workspace_dev, size_t ws_bytes, int32_t* status_dev, void* stream) {
  if (!pooled_dev) return DSF_EINVAL;
  return run_attention(tables, kjt, seq, q_feat, seq_table, B, mlp, pooled_dev, din_dev, logits_dev,
                       workspace_dev, ws_bytes, status_dev, stream);
}

const char* dsf_status_string(int code) {
  switch (code) {
    case DSF_OK: return "ok";
    case DSF_EINVAL: return "invalid argument";
    case DSF_EUNSUPPORTED: return "unsupported configuration";
    case DSF_ECUDA: return "CUDA error";
    case DSF_EWORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

int dsf_read_status(const int32_t* status_dev, int32_t* status_host, void* stream) {
  if (!status_dev || !status_host) return DSF_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, status_dev, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return DSF_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSF_ECUDA;
  *status_host = v;
  return DSF_OK;
}

int32_t dsf_grid_size(int32_t D, int32_t dtype, int32_t mode, int32_t with_attention) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const bool bf16 = dtype == DSF_BF16;
  if (!with_attention) return grid_pool(D, bf16, dev);
  if (mode == DSF_MODE_BF16_TC) return grid_attn_tc(D, bf16, dev);
  return grid_attn_f32(D, bf16, dev);
}

// ---------------------------------------------------------------------------
// EmbeddingBag pooling without a caller workspace.
//
// For callers that cannot allocate device memory, e.g. a serving runtime whose
// device memory is owned by its own arena allocator, or code that runs while a
// stream is being captured, where cudaMalloc is not allowed. The pooling
// kernel's only scratch is the exchange state (workspace header plus the
// per-CTA partial sums); here it lives in one fixed array compiled into the
// library instead. Host code must not use the array's name as a device
// address: its address is looked up per device at first use.

}  // extern "C"

namespace dsf {
namespace {

// Header + partials for up to kMaxG CTAs x kMaxF tables: 262,400 bytes held on
// every device that loads the library, until the process exits.
constexpr size_t kStaticScratchBytes = kWsWpackOff;
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, cleared on the
// first call for that device (the clear is queued on `stream`).
int static_scratch(int dev, cudaStream_t stream, void** out) {
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return DSF_ECUDA;
    if (cudaMemsetAsync(ptr, 0, kStaticScratchBytes, stream) != cudaSuccess) return DSF_ECUDA;
    g_static_ptr[dev] = ptr;
  }
  *out = g_static_ptr[dev];
  return DSF_OK;
}

}  // namespace
}  // namespace dsf

extern "C" {

int emb_bag_pool_noalloc(const dsf_tables* tables, const dsf_kjt* kjt, int32_t B,
                         float* pooled_dev, int32_t* status_dev, void* stream) {
  int rc;
  if ((rc = check_tables(tables)) != DSF_OK) return rc;
  if (B < 0 || B > (1 << 24)) return DSF_EINVAL;
  if ((rc = check_kjt(kjt, B, tables->F)) != DSF_OK) return rc;
  if (!pooled_dev || !aligned(pooled_dev, 16)) return DSF_EINVAL;
  if (B == 0) return DSF_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSF_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return DSF_EUNSUPPORTED;
  const bool bf16 = tables->dtype == DSF_BF16;
  // (the pooling grid is capped at the scratch's tagged words, one per CTA)
  if (grid_pool(tables->D, bf16, dev) <= 0) return DSF_EUNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  if ((rc = static_scratch(dev, s, &scratch)) != DSF_OK) return rc;
  FwdParams p;
  fill_common(p, tables, kjt, B, scratch, status_dev);
  p.pooled = pooled_dev;
  p.max_len = 1;
  return map_launch(launch_pool(tables->D, bf16, p, s));
}

}  // extern "C"
