/*
 * dinsparse.h -- C ABI of the GB300 (sm_103a) MultiTowerDIN sparse forward.
 *
 * The path computes, for a batch of B samples:
 *   (a) EmbeddingBag sum pooling of a KeyedJaggedTensor over F tables:
 *       pooled[b, f*D:(f+1)*D] = sum of table_f rows over bag (f, b).
 *       ("MultiTowerDIN: current state analysis", section 3: one [num_buckets, 16]
 *       table per id feature, sum-pooled lookup; section 2: SparseData(values,
 *       lengths) becomes a KeyedJaggedTensor.)
 *   (b) Padding-free DIN target attention:
 *       q_b    = cat of the pooled bags of the three target features
 *                (adgroup_id / cate_id / brand; section 1 feature groups),
 *       s_b,t  = cat of the three sequence sub-feature rows at position t,
 *                read from the same tables ("MultiTowerDIN: integrating
 *                DynamicEmb", section 2.4: shared embedding tables),
 *       x      = cat[q, s, q - s, q * s]          (section 4.2 code block),
 *       z      = w3 . ReLU(W2 ReLU(W1 x + b1) + b2) + b3
 *                (attn_mlp hidden [256, 64], then a linear to 1; section 4.2),
 *       a      = softmax of z over the valid positions t < L_b only
 *                (section 4.2 mask + softmax; the padding to max_len that the
 *                pages' flow builds is never materialised here),
 *       din[b] = sum_t a_t s_b,t                 (section 4.4 weighted sum).
 *
 * Conventions for every entry point:
 *   - All pointers named *_dev or documented "device" are device pointers
 *     (CUDA global memory); all others are host pointers. Every device buffer
 *     is allocated and freed by the caller; the library never allocates.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls are asynchronous on it. The return value covers argument checks and
 *     launch errors only; data errors found on the device are OR-ed into
 *     *status_dev (DSF_FLAG_* bits), which the caller zeroes beforehand.
 *   - One workspace may serve one stream at a time: two calls that overlap on
 *     the GPU must not share a workspace (its launch epoch and per-block
 *     partial sums would race).
 *   - The library keeps per-device state from its first call on a device
 *     (grid sizes, the address of emb_bag_pool_noalloc's array, library
 *     handles). It does not survive cudaDeviceReset of that device: after a
 *     reset, start a new process before calling it again.
 *   - Device data errors never fault or trap: an id outside [0, rows) or a
 *     value index past the values array contributes a zero row; a negative
 *     length counts as zero; a sequence longer than max_len keeps its first
 *     max_len positions. Each sets its flag bit.
 */
#ifndef DINSPARSE_H
#define DINSPARSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSF_MAX_TABLES 32

/* Table element types. */
enum { DSF_F32 = 0, DSF_BF16 = 1 };

/* Attention-MLP arithmetic. BF16_TC: bf16 operands on tcgen05 tensor cores,
 * fp32 accumulation (the pages' half-precision MLP, "integrating DynamicEmb",
 * section 3.3). FP32: fp32 CUDA-core arithmetic, a check mode. */
enum { DSF_MODE_BF16_TC = 0, DSF_MODE_FP32 = 1 };

/* Return codes. */
enum {
  DSF_OK = 0,
  DSF_EINVAL = 1,        /* null pointer, bad size, index out of range ... */
  DSF_EUNSUPPORTED = 2,  /* a D / dtype / MLP shape this library does not build */
  DSF_ECUDA = 3,         /* a CUDA runtime call or kernel launch failed */
  DSF_EWORKSPACE = 4     /* workspace missing, too small or misaligned */
};

/* Bits OR-ed into *status_dev by the kernels. */
#define DSF_FLAG_ID_RANGE      0x01 /* an id outside [0, rows) (contributes zero) */
#define DSF_FLAG_NEG_LENGTH    0x02 /* a negative length (counted as zero) */
#define DSF_FLAG_SEQ_TRUNC     0x04 /* a sequence longer than max_len was cut */
#define DSF_FLAG_COUNT         0x08 /* lengths sum differs from the values array size */
#define DSF_FLAG_TIMEOUT       0x10 /* a device wait ran out (about 1 s); outputs invalid */
#define DSF_FLAG_NOT_PREPARED  0x20 /* dsf_prepare_mlp was not run on this workspace */
#define DSF_FLAG_HASH          0x40 /* the hash workspace was not initialised for this capacity */
#define DSF_FLAG_HASH_FULL     0x80 /* dsf_hash_insert found no free slot for a key (left out) */
#define DSF_FLAG_GRAD_LIST     0x100 /* more touched rows than the row-gradient list holds */

/* Pooling of a table's bags (EmbeddingBag modes: the pages' tables pool by
 * sum, section 3; mean divides the fp32 sum by the bag's length, an empty bag
 * staying 0). */
#define DSF_POOL_SUM  0
#define DSF_POOL_MEAN 1

/* ------------------------------------------------------------------------
 * Hash-table storage for large tables (MultiTowerDIN: integrating DynamicEmb,
 * sections 1 and 3.2: open-addressing hash lookup; the large tables of a
 * feature group fused into one storage with independent key spaces; an unseen
 * id reads the constant 0). Admission and eviction are not part of this
 * library: keys and their rows are inserted by the caller.
 *
 * A table served this way takes raw ids in [0, 2^56) as keys in its own key
 * space (0 .. 254), so equal raw ids of two tables never collide. Several
 * tables share one workspace: one key array (buckets of 8 slots, one 64-byte
 * line each, probed linearly from a 64-bit hash of the key) and one row pool
 * [slots + 1, D] whose last row is zero.
 *
 * workspace: device, 256-byte aligned, dsf_hash_workspace_bytes(capacity, D,
 * dtype) bytes, caller-owned. capacity: the minimum slot count (rounded up to
 * 8 times a power of two); keep the keys at most ~3/4 of it. key_space: host
 * array [F] for dsf_tables (-1: table f is a plain table; k: table f's ids are
 * raw keys of key space k), unused by the calls below. */
typedef struct {
  void* workspace;
  size_t ws_bytes;
  int64_t capacity;
  int32_t D;      /* 16 or 64, as the tables it serves */
  int32_t dtype;  /* DSF_F32 or DSF_BF16 */
  const int32_t* key_space;
} dsf_hash;

/* Bytes of a hash workspace (0 for invalid arguments). */
size_t dsf_hash_workspace_bytes(int64_t capacity, int32_t D, int32_t dtype);

/* Empties the table: every slot free, the zero row zeroed, the header written.
 * Asynchronous on stream. */
int dsf_hash_init(const dsf_hash* hash, void* stream);

/* Inserts n keys (device int64 [n], raw ids in [0, 2^56)) of one key space
 * with their rows (device [n, D] of the table dtype, 16-byte aligned). A key
 * already present has its row overwritten; a key given twice in one call keeps
 * one of its rows. A raw id out of range sets DSF_FLAG_ID_RANGE, a key with no
 * free slot DSF_FLAG_HASH_FULL, an uninitialised workspace DSF_FLAG_HASH (in
 * *status_dev, nullable); those keys are left out. Asynchronous on stream. */
int dsf_hash_insert(const dsf_hash* hash, int32_t key_space, const int64_t* keys_dev, const void* rows_dev,
                    int64_t n, int32_t* status_dev, void* stream);

/* The lookup alone: slots_dev[i] = the slot of keys_dev[i] in key_space, the
 * zero row's index (the slot count) for an unseen key, or -2 (with
 * DSF_FLAG_ID_RANGE) for a raw id outside [0, 2^56). Device int64 arrays [n]. */
int dsf_hash_find(const dsf_hash* hash, int32_t key_space, const int64_t* keys_dev, int64_t n, int64_t* slots_dev,
                  int32_t* status_dev, void* stream);

/* F embedding tables, one per KJT key, all with the same D and element type.
 * table_ptrs[f]: device pointer to a row-major [table_rows[f], D] table,
 * 16-byte aligned. Host arrays of length F. pooling: host array [F] of
 * DSF_POOL_SUM / DSF_POOL_MEAN, or NULL for all sum. A mean-pooled query
 * table feeds the attention its mean too. hash: NULL, or the hash-table
 * storage serving the tables whose hash->key_space[f] >= 0 (their table_ptrs
 * and table_rows entries are then ignored; an unseen key adds a zero row and
 * counts in a mean's length; a raw id outside [0, 2^56) sets
 * DSF_FLAG_ID_RANGE and adds nothing). Its D and dtype match the tables'. */
typedef struct {
  const void* const* table_ptrs;
  const int64_t* table_rows;
  int32_t F;      /* 1 .. DSF_MAX_TABLES */
  int32_t D;      /* 16 or 64 */
  int32_t dtype;  /* DSF_F32 or DSF_BF16 */
  const int32_t* pooling;
  const dsf_hash* hash;
} dsf_tables;

/* KeyedJaggedTensor of the deep group (section 2: values + lengths).
 * lengths_dev: int32 [F*B], key-major (the B bags of key 0, then key 1 ...);
 * values_dev: int64 [n_values], the row ids of all bags in the same order. */
typedef struct {
  const int64_t* values_dev;
  int64_t n_values;
  const int32_t* lengths_dev;
} dsf_kjt;

/* The behaviour sequence (section 2: SequenceSparseData(values, seq_lengths)).
 * values_dev: int64 [3, n_per_key], key-major: sub-feature k's ids are
 * values_dev[k*n_per_key + j]; the positions of sample b are
 * j = seq_off[b] .. seq_off[b] + L_b - 1 with seq_off the exclusive scan of
 * lengths_dev (int32 [B]). max_len: the sequence cap (section 4.1, 100). */
typedef struct {
  const int64_t* values_dev;
  int64_t n_per_key;
  const int32_t* lengths_dev;
  int32_t max_len;
} dsf_seq;

/* The attention MLP, device fp32, PyTorch Linear layout [out, in]:
 * W1 [N1, K1], b1 [N1], W2 [N2, N1], b2 [N2], w3 [N2], b3 [1].
 * K1 = 4 * 3 * D, N1 = 256, N2 = 64 (attn_mlp hidden_units [256, 64]). */
typedef struct {
  const float *W1, *b1, *W2, *b2, *w3, *b3;
  int32_t K1, N1, N2;
  int32_t mode; /* DSF_MODE_BF16_TC or DSF_MODE_FP32 */
} dsf_mlp;

/* Bytes of workspace needed for batch size B and embedding dim D (packed MLP
 * weights, epoch-tagged per-block partial sums, launch epoch, query buffer).
 * Returns 0 for unsupported D. */
size_t dsf_workspace_bytes(int32_t B, int32_t D);

/* Zeroes the workspace's exchange state (launch epoch and tagged partial
 * sums). Call once after allocating a workspace, before any other call that
 * uses it, and again after a call reported DSF_FLAG_TIMEOUT. Asynchronous on
 * stream. */
int dsf_workspace_init(void* workspace_dev, size_t ws_bytes, void* stream);

/* Packs the MLP weights into the workspace: bf16 in the tensor-core operand
 * layout (128-byte swizzled, K-major) and fp32 transposed copies for the check
 * mode. Call again whenever W1 / W2 change; b1, b2, w3, b3 are read directly at
 * each forward call. D selects the shape (K1 = 12 * D). */
int dsf_prepare_mlp(const dsf_mlp* mlp, int32_t D, void* workspace_dev, size_t ws_bytes,
                    void* stream);

/* (a) EmbeddingBag sum pooling of all F keys.
 * pooled_dev: fp32 [B, F*D], row-major; bag (f, b) goes to columns
 * [f*D, (f+1)*D). Each bag is summed in fp32 in value order (an empty bag
 * gives zeros). B >= 0; B = 0 is a no-op. */
int emb_bag_pool(const dsf_tables* tables, const dsf_kjt* kjt, int32_t B, float* pooled_dev,
                 void* workspace_dev, size_t ws_bytes, int32_t* status_dev, void* stream);

/* (b) Jagged DIN target attention.
 * q_feat[3]: KJT keys whose pooled bags form the query (target items).
 * seq_table[3]: table index of each sequence sub-feature.
 * din_dev: fp32 [B, 3*D]; a sample with no valid position gets zeros.
 * logits_dev (nullable): fp32 [n_per_key]; receives z for every valid position
 * j of the sequence values (positions past max_len are left untouched). */
int din_jagged_attn(const dsf_tables* tables, const dsf_kjt* kjt, const dsf_seq* seq,
                    const int32_t q_feat[3], const int32_t seq_table[3], int32_t B,
                    const dsf_mlp* mlp, float* din_dev, float* logits_dev,
                    void* workspace_dev, size_t ws_bytes, int32_t* status_dev, void* stream);

/* (a) + (b) in one launch: pooled_dev as emb_bag_pool, din_dev as
 * din_jagged_attn, with the query read from the pooled rows. */
int din_sparse_fwd(const dsf_tables* tables, const dsf_kjt* kjt, const dsf_seq* seq,
                   const int32_t q_feat[3], const int32_t seq_table[3], int32_t B,
                   const dsf_mlp* mlp, float* pooled_dev, float* din_dev, float* logits_dev,
                   void* workspace_dev, size_t ws_bytes, int32_t* status_dev, void* stream);

/* (a) EmbeddingBag sum pooling, as emb_bag_pool, for callers that cannot
 * allocate device memory -- for instance a serving runtime whose device memory
 * belongs to its own arena allocator, or code that runs inside a stream
 * capture, where cudaMalloc is not permitted. The pages have no counterpart to
 * this entry point; it exists only for such callers.
 * It takes no workspace: the cross-CTA exchange state (a header and one partial
 * sum per CTA and table) lives in a fixed 262,400-byte array compiled into the
 * library, which every GPU that loads the library holds until the process
 * exits. Limits: F <= DSF_MAX_TABLES (32); the pooling grid is capped at
 * 32,768 CTAs (one tagged word each in the array), far above any device's
 * resident CTAs; B is not limited by the array.
 * The first call on a device, made with that device current, looks up the
 * array's device address and clears it on `stream`; make that first call
 * before any stream capture (later calls may be captured into a graph and
 * replayed). Every call shares the one array and leaves it ready for the next
 * call, so calls that overlap on the GPU (for instance on two streams) race:
 * serialise them. After a call that set DSF_FLAG_TIMEOUT, that call's pooled
 * rows are invalid; the array needs no reset, since the kernel advances its
 * launch epoch on a timeout as well and the next call's exchange starts from
 * it. Allocates nothing (no cudaMalloc or cudaFree, no allocating library
 * call). */
int emb_bag_pool_noalloc(const dsf_tables* tables, const dsf_kjt* kjt, int32_t B,
                         float* pooled_dev, int32_t* status_dev, void* stream);

/* Human-readable name of a return code. */
const char* dsf_status_string(int code);

/* Copies the status word *status_dev (the DSF_FLAG_* bits the calls on
 * `stream` OR-ed into it) to *status_host once the work queued on `stream`
 * before this call has finished: an asynchronous device-to-host copy on
 * `stream`, then a wait for that stream (blocks the host thread). The pages
 * define no such call; it is the host side of the status convention above.
 * Returns DSF_EINVAL for a null pointer (nothing copied), DSF_ECUDA if the
 * copy or the wait fails (*status_host unchanged); must not be called while
 * `stream` is being captured into a graph. */
int dsf_read_status(const int32_t* status_dev, int32_t* status_host, void* stream);

/* Grid size (CTAs) the forward kernels use on the current device for this
 * call shape; 0 if unsupported. For diagnostics and benchmarks. */
int32_t dsf_grid_size(int32_t D, int32_t dtype, int32_t mode, int32_t with_attention);

/* ------------------------------------------------------------------------
 * The dense towers after the sparse path (MultiTowerDIN: current state
 * analysis, section 4.4; the model config, section 7): the deep tower
 * h = ReLU(Wd3 ReLU(Wd2 ReLU(Wd1 p + bd1) + bd2) + bd3) on the pooled deep
 * group p [256] (widths 512, 256, 128) and the final tower
 * logit = wo . ReLU(Wf1 cat[h, din] + bf1) + bo on cat[h, din] [176]. The
 * GEMMs take bf16 operands (inputs rounded to nearest-even bf16 after bias
 * and ReLU in fp32) and accumulate in fp32 on the tensor cores.
 *
 * Device fp32 weights in Linear [out, in] layout: Wd1 [512, 256], bd1 [512],
 * Wd2 [256, 512], bd2 [256], Wd3 [128, 256], bd3 [128], Wf1 [64, 176],
 * bf1 [64], wo [64], bo [1]. The biases, wo and bo are read at each call;
 * the four matrices are packed into the towers workspace by
 * dsf_prepare_towers (call again when they change). */
typedef struct {
  const float *Wd1, *bd1, *Wd2, *bd2, *Wd3, *bd3;
  const float *Wf1, *bf1, *wo, *bo;
} dsf_towers;

/* Bytes of the towers workspace (packed bf16 weights and a prepared tag);
 * the caller allocates it, 256-byte aligned. */
size_t dsf_towers_workspace_bytes(void);

/* Packs the tower matrices into the workspace (asynchronous on stream). */
int dsf_prepare_towers(const dsf_towers* towers, void* workspace_dev, size_t ws_bytes, void* stream);

/* The towers on the outputs of din_sparse_fwd (D = 16): pooled_dev [B, 256]
 * and din_dev [B, 48] fp32, 16-byte aligned; writes logit_dev [B] fp32. One
 * 512-thread CTA per 128 samples. Returns DSF_EWORKSPACE for a missing or
 * small workspace; DSF_FLAG_NOT_PREPARED when dsf_prepare_towers has not run
 * on it; DSF_FLAG_TIMEOUT if a device wait ran out. */
int ctr_towers_fwd(const float* pooled_dev, const float* din_dev, int32_t B, const dsf_towers* towers,
                   float* logit_dev, const void* workspace_dev, size_t ws_bytes, int32_t* status_dev,
                   void* stream);

/* ------------------------------------------------------------------------
 * Backward of the sparse path and the sparse optimizer step (MultiTowerDIN:
 * current state analysis, section 1: training with sparse AdaGrad, lr 1e-3;
 * the forward of sections 4.2 and 4.4 differentiated).
 *
 * din_sparse_bwd takes the forward's inputs, its pooled output and the
 * upstream gradients dpooled [B, F*D] (nullable: zero) and ddin [B, 3D]
 * (fp32, device, 16-byte aligned), recomputes the attention forward, and
 * produces
 *   - the attention MLP's gradients (dsf_mlp_grads, device fp32, overwritten:
 *     dW1 [256, 12D], db1 [256], dW2 [64, 256], db2 [64], dw3 [64], db3 [1]);
 *   - every touched row's summed gradient, accumulated into dsf_row_grads.
 * The MLP runs as in the forward's mode (mlp->mode): bf16 GEMM operands with
 * fp32 accumulation, or fp32 throughout. Its six matrix products are this
 * library's GEMMs (tcgen05 tensor cores fed by TMA for bf16 operands, CUDA
 * cores in the fp32 mode) over the sequence values' length (rows past the
 * valid count are zero), with the ReLU, the mask and (at D = 16) ds fused
 * into their epilogues; the rest are this library's kernels. Row gradients are summed with
 * fp32 atomics, so their rounding order varies between runs. Gradients of
 * unseen hash keys and of invalid ids are dropped. emb_adagrad_update then
 * applies AdaGrad to the touched rows and leaves the row-gradient state zero
 * for the next step.
 *
 * Row-gradient state, caller-owned: host arrays [F] of device pointers, per
 * table f: grad[f] fp32 [rows_f, D] and touched[f] int32 [rows_f], zero
 * before the first step; for the tables served by a hash table, the pool's
 * [slots + 1, D] and [slots + 1] arrays, the same pointers for all of them.
 * list: device int64 [list_cap], the touched rows (table << 40 | row); count:
 * device int32 [1], zero before the first step. list_cap bounds the distinct
 * rows of one step (at most n_values + 3 * n_per_key); more set
 * DSF_FLAG_GRAD_LIST. */
typedef struct {
  float *dW1, *db1, *dW2, *db2, *dw3, *db3;
} dsf_mlp_grads;

typedef struct {
  float* const* grad;
  int32_t* const* touched;
  int64_t* list;
  int32_t* count;
  int64_t list_cap;
} dsf_row_grads;

/* Workspace bytes of din_sparse_bwd for B samples, n_values KJT values and
 * n_per_key sequence values (0 for invalid arguments); caller-owned,
 * 256-byte aligned. */
size_t dsf_bwd_workspace_bytes(int32_t B, int64_t n_values, int64_t n_per_key, int32_t D);

/* Where din_sparse_bwd leaves its per-position intermediates inside a
 * workspace sized by dsf_bwd_workspace_bytes with the same arguments: byte
 * offsets from the workspace's start, written to offsets[6] in this order
 *   x   [P, 12D] MLP operand type    [q, s, q - s, q * s] per position
 *   h1  [P, 256] MLP operand type    ReLU(x W1^T + b1)
 *   h2  [P, 64]  fp32                h1 W2^T (b2 not added)
 *   dh2 [P, 64]  MLP operand type    dz w3 [h1 W2^T + b2 > 0]
 *   g   [P, 256] fp32                dh2 W2 (before the layer-1 mask)
 *   dh1 [P, 256] MLP operand type    g [h1 > 0]
 * (operand type: bf16 in DSF_MODE_BF16_TC, else fp32; rows: the valid
 * sequence positions in sample order, then zero rows up to n_per_key). The
 * values stay there from the end of a din_sparse_bwd call on that workspace
 * until the workspace's next use. An inspection aid (for tests of the
 * intermediate values): the pages define no such call. Host only, no CUDA
 * call; DSF_EINVAL for a null pointer or arguments that
 * dsf_bwd_workspace_bytes rejects. */
int dsf_bwd_workspace_offsets(int32_t B, int64_t n_values, int64_t n_per_key, int32_t D, int64_t* offsets);

/* Returns DSF_EINVAL / DSF_EUNSUPPORTED / DSF_EWORKSPACE for bad arguments
 * (as din_sparse_fwd), DSF_ECUDA when a launch or a CUDA call fails (the
 * products' TMA tensor maps are encoded through the driver at each call).
 * Device data errors set bits in *status_dev (nullable). Asynchronous on
 * stream, in this workspace: steps that no next step needs run on a second
 * stream of the library's (one per device, made by the first call that is
 * not being captured into a CUDA graph), forked from and joined back to
 * `stream` by events before the call returns; a captured call records that
 * fork and join, or, with no second stream yet, runs every step on
 * `stream`. */
int din_sparse_bwd(const dsf_tables* tables, const dsf_kjt* kjt, const dsf_seq* seq,
                   const int32_t* q_feat, const int32_t* seq_table, int32_t B, const dsf_mlp* mlp,
                   const float* pooled_dev, const float* dpooled_dev, const float* ddin_dev,
                   const dsf_mlp_grads* mlp_grads, const dsf_row_grads* row_grads, void* workspace_dev,
                   size_t ws_bytes, int32_t* status_dev, void* stream);

/* Sparse AdaGrad on the touched rows: per element G += g * g and
 * w -= lr * g / (sqrt(G) + eps), in fp32 (bf16 tables round the new weight to
 * nearest even); then the rows' gradients, touched flags and the count are
 * zeroed. The tables (their table_ptrs, or the hash pool) are updated in
 * place. accum: host array [F] of device fp32 [rows_f, D] AdaGrad
 * accumulators (the pool's for hash-table tables, as for the gradients). */
int emb_adagrad_update(const dsf_tables* tables, float* const* accum, const dsf_row_grads* row_grads, float lr,
                       float eps, int32_t* status_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DINSPARSE_H */
