// Host/device declarations shared by the translation units of libgrpo.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "grpo.h"

namespace grpo {

// Device-side index checks of the checked build (compiled with
// GRPO_DEVICE_CHECKS): GRPO_DCHECK(cond, status) is cond, and a false cond
// also records GRPO_ERR_BOUNDS in the caller's status word; the caller then
// skips the access.  In the normal build it is the constant true and costs
// nothing.  The checks cover every global index a kernel takes from device
// data (the valid-row list) and the offset arithmetic of the chunk buffers.
#ifdef GRPO_DEVICE_CHECKS
__device__ inline bool dcheck(bool ok, int* status) {
    if (!ok) atomicCAS(status, 0, GRPO_ERR_BOUNDS);
    return ok;
}
#define GRPO_DCHECK(cond, status) ::grpo::dcheck((cond), (status))
#else
#define GRPO_DCHECK(cond, status) true
#endif

constexpr int kBM = 128;              // rows (or vocabulary rows for dW) per MMA tile
constexpr int kBK = 64;               // K elements per pipeline stage: one 128-byte swizzle span
constexpr int kBN = 256;              // accumulator columns per MMA tile
constexpr int kTileSplits = 8;        // vocabulary splits of a forward row tile (forward-only path)
constexpr int kChunkSplits = 64;      // vocabulary splits of a chunk row tile (forward+backward path), target
constexpr int kChunkSplitsMax = 256;  // ... and the most it may take to divide the vocabulary tiles evenly
// Default rows per backward chunk, in 128-row tiles: the smaller of 38 and 76
// whose dH units ((tiles / 2) tile pairs x ceil(d / 256) d tiles) divide
// evenly over the 76 SM pairs of a GB300 (38 for d = 4096 or 5120, 76 for
// d = 1536).  Smaller chunks than that leave dH a part-empty last wave; larger
// ones hold more dlogits memory and ran slower (a larger, busier working set
// under the power cap).
constexpr int kChunkPairs = 76;
constexpr int kChunkTilesSmall = 38;
constexpr int kChunkTilesLarge = 76;
constexpr int kMergeThreads = 256;
constexpr int kIndexThreads = 1024;
constexpr int kTransformThreads = 256;

// int32 words at the start of the workspace
enum CountSlot {
    C_NVALID = 0,      // masked-in rows
    C_NTILES = 1,      // forward row tiles
    C_NCHUNKS = 2,     // backward chunks
    C_CHUNK_ROWS = 3,  // rows per backward chunk (multiple of 128)
    C_WINV = 4,        // 1 / max(N_div, 1) as float bits: the weight of one row in the token mean
    C_NACT = 5,        // completions with at least one masked-in row
    C_SHARD = 6,       // 1 when the divisors below come from the caller's global counts (a data-parallel shard)
    C_NDIV_G = 7,      // shard: masked-in rows over all shards (the token mean's divisor)
    C_NACT_G = 8,      // shard: completions with a masked-in row over all shards (the sequence mean's divisor)
    C_SPARE_INF = 9,   // found_inf word of the 8-bit backward, which has no loss scaling
    C_COUNT_WORDS = 16
};

// divisors of the mean: this call's own counts, or the global ones of a shard
__device__ __forceinline__ int count_ndiv(const int* counts) {
    return counts[C_SHARD] ? counts[C_NDIV_G] : counts[C_NVALID];
}
__device__ __forceinline__ int count_nact(const int* counts) {
    return counts[C_SHARD] ? counts[C_NACT_G] : counts[C_NACT];
}

// The 8-bit backward sorts each chunk's (token, slot) keys in one block's
// shared memory: chunks of at most this many rows.
constexpr int kF8SortMax = 16384;

struct WsLayout {
    size_t counts, sched, seqcnt, tiles, rows, part, zt, lse, gco, ell, blocksum, hc, hcr, partc, mx, ds, total;
    // 8-bit inputs only (grpo_loss_fwd_bwd_fp8): row maxima [N] f32, the two code
    // buffers of the softmax part of the dlogits [R x V_pad] u8 each, the group
    // scales [nc32] f32, every chunk's sorted (token, slot) keys [max chunks x R]
    // u64 and the first key of each token in the current chunk [V] i32
    size_t rmax, qa, qb, gmax, keys, tokpos;
    size_t hct;      // the chunk's compact h_pol rows transposed, [d x R] 16-bit (dW's K-major B operand)
    int S, nps;      // forward-only path: vocabulary splits, N-tiles per split (partials by row)
    int Sc, npsc;    // chunked path: vocabulary splits, N-tiles per split (partials by chunk slot)
    int n_ntiles;    // ceil(V / kBN)
    int R;           // rows per backward chunk (buffer height)
    int V_pad;       // row pitch of the dlogits buffer, elements
    int nc32;        // row pitch of the running maxima: 32-column groups per vocabulary row, rounded up to 8
    int nblk;        // loss-reduction blocks
    int n_sched;     // scheduler counters
    int n_seq;       // completions (n_groups * G)
    int64_t N;
};

bool ws_layout(const grpo_shape& s, WsLayout* out);
inline bool is_fp8(grpo_dtype t) { return t == GRPO_E4M3 || t == GRPO_E5M2; }

// Forward logits + streaming logsumexp.  Two row sources:
//   tiles != nullptr : forward row tiles over h_pol / h_ref (runs of masked-in rows)
//   tiles == nullptr : the compact rows of backward chunk `chunk` (gathered copies);
//                      then E/mx receive exp(z_pol - running max) and the running max
struct FwdParams {
    const int2* tiles;      // (first row, rows) per forward tile, or nullptr
    const int* counts;
    const int* rows;        // valid-row list (chunk mode)
    const int* tokens;
    float4* part;           // (m_pol, s_pol, m_ref, s_ref): [N x S] by row, or [R x S] by chunk slot
    float2* zt;             // [N] (z_pol[tok], z_ref[tok])
    uint16_t* E;            // [R x V_pad] bf16 exp(z_pol - m) (chunk mode, may be nullptr)
    float* mx;              // [R x nc32] running max after each 32-column group (chunk mode)
    int* sched;             // zeroed work counter of this launch
    float zscale[2];        // logits = zscale * accumulator (policy, reference); 1 unless 8-bit inputs
    int64_t N;
    int chunk;
    int V, d, S, nps, n_ntiles, V_pad, nc32;
    int R;                  // chunk mode: rows of the chunk buffers (index checks)
    int* status;
};

struct ChunkParams {
    const int* counts;
    const int* rows;        // valid-row list
    const int* tokens;
    const float* lse;       // [N] policy logsumexp
    const float* gco;       // [N] d ell / d q
    const float2* zt;       // [N] (z_pol[tok], z_ref[tok])
    const float* mx;        // [R x nc32]
    float scale;            // loss scale
    int chunk;
    int V, d, V_pad, nc32;
    int R;                  // rows of the chunk buffers
    int64_t N;              // rows of h_pol / dH (index checks)
    uint16_t* dS;           // [R x V_pad] scaled dlogits (without the 1/N_valid factor)
    uint16_t* dH;           // [N x d]
    float* dW;              // [V x d]
    int* sched;             // zeroed work counter of this launch
    int* found_inf;
    int* status;
    // 8-bit backward: P = g * softmax (the dlogits without their one-hot part) as
    // 8-bit codes, scaled per row (qa, for dH) and per 32-column group (qb, for dW)
    uint8_t* qa;            // [R x V_pad]  P * 448 / (|g| max_v softmax) of the row
    uint8_t* qb;            // [R x V_pad]  P * 448 / gmax[group]
    const float* rmax;      // [N] row maximum of the policy logits
    float* gmax;            // [nc32] max over the chunk's rows of |P| bounds per 32-column group
    unsigned long long* keys;   // (token << 32 | slot) of the chunk's rows, ascending: [R] of this chunk
                                //   (the sort writes every chunk's, [max chunks x R], from the first chunk's base)
    int* tokpos;            // [V] index in keys of the token's first key, -1 if no row of the chunk has it
    const uint8_t* hq;      // compact 8-bit h_pol rows of the chunk [R x d]
    const uint8_t* wq;      // 8-bit W [V x d]
    float scale_h, scale_w; // per-tensor scales of the 8-bit h_pol and W
    int e5m2;               // code format: E5M2 (1) or E4M3 (0)
};

struct MergeParams {
    const float4* part;     // [N x S] by row (chunk < 0), or [R x S] by chunk slot
    const float2* zt;
    const uint8_t* mask;
    const int* tokens;
    const float* adv;
    const int* counts;
    const int* rows;        // chunk mode: valid-row list
    int chunk;              // < 0: every row t in [0, N)
    int R;                  // chunk rows (buffer height)
    int S, L, V;
    float beta;
    int loss_mode;          // GRPO_TOKEN_MEAN / GRPO_SEQUENCE_MEAN
    int objective;          // GRPO_OBJ_*
    const int* seqcnt;      // masked-in rows per completion
    int64_t N;
    float* lse;
    float* gco;
    float* ell;
    float* row_stats;
    int* status;
    float* rmax;            // nullable: row maximum of the policy logits (the 8-bit backward)
};

// ---- launches (return cudaError_t of the launch) ----
cudaError_t launch_index(const uint8_t* mask, int64_t N, int R_max, int* counts, int* rows, int2* tiles,
                         int* sched, int n_sched, int* status, cudaStream_t st);
cudaError_t launch_advantages(const float* r, int n_groups, int G, float eps, int std_unbiased, float* adv,
                              cudaStream_t st);
cudaError_t launch_build_mask(const int32_t* lengths, int n_seq, int L, uint8_t* mask, cudaStream_t st);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t st);
cudaError_t launch_seq_counts(const uint8_t* mask, int n_seq, int L, int* seqcnt, int* counts, cudaStream_t st);
// data-parallel shards: this shard's (masked-in rows, active completions), and the
// switch of the divisors to the caller's global counts
cudaError_t launch_shard_counts(const uint8_t* mask, int n_seq, int L, int* out, cudaStream_t st);
cudaError_t launch_apply_global_counts(const int* global_counts, int* counts, int loss_mode, int* status,
                                       cudaStream_t st);
cudaError_t launch_rows_init(const uint8_t* mask, int64_t N, float* ell, float* row_stats, int sm_count,
                             cudaStream_t st);
cudaError_t launch_loss_reduce(const float* ell, int64_t N, double* blocksum, int nblk, const int* counts,
                               float* loss_out, cudaStream_t st);
// The grid-stride kernels below size their grids in multiples of the device's SM count.
cudaError_t launch_gather_rows(const ChunkParams& p, const void* h_pol, void* hc, const void* h_ref, void* hcr, int R,
                               int row_bytes, int sm_count, cudaStream_t st);
// 16-bit inputs: the same gather, also writing the transpose of the compact h_pol rows
cudaError_t launch_gather_rows_t(const ChunkParams& p, const void* h_pol, void* hc, const void* h_ref, void* hcr,
                                 void* hct, int R, int sm_count, cudaStream_t st);
cudaError_t launch_transform(const ChunkParams& p, bool bf16, int R, int sm_count, cudaStream_t st);
cudaError_t launch_clear_grads(const int* counts, int* found_inf, float* dW, int64_t n, int sm_count, cudaStream_t st);
cudaError_t launch_zero_masked_rows(const uint8_t* mask, int64_t N, int d, void* dH, int sm_count, cudaStream_t st);
// 8-bit backward: group bounds, dlogit codes, sorted token keys, and the two GEMMs
cudaError_t launch_f8_group_max(const ChunkParams& p, int sm_count, cudaStream_t st);
cudaError_t launch_transform_f8(const ChunkParams& p, int sm_count, cudaStream_t st);
cudaError_t launch_sort_keys(const ChunkParams& p, int max_chunks, cudaStream_t st);

cudaError_t launch_wait_selftest(int* status, unsigned long long* waited_ns, cudaStream_t st);
#ifdef GRPO_DEVICE_CHECKS
cudaError_t launch_bounds_selftest(int* status, cudaStream_t st);
#endif
cudaError_t launch_fwd(const FwdParams& p, const CUtensorMap& mHp, const CUtensorMap& mHr,
                       const CUtensorMap& mW, int n_sm, bool bf16, cudaStream_t st);
// CTA-pair (M=256) variants: forward of a chunk, dH, dW
cudaError_t launch_fwd_pair(const FwdParams& p, const CUtensorMap& mHp, const CUtensorMap& mHr,
                            const CUtensorMap& mW, int n_sm, bool bf16, cudaStream_t st);
cudaError_t launch_fwd_pair_fp8(const FwdParams& p, const CUtensorMap& mHp, const CUtensorMap& mHr,
                                const CUtensorMap& mW, int n_sm, bool e5m2, cudaStream_t st);
// wide: 512-column units (see DhPairWideT), for chunks whose wide units divide evenly over the SM pairs
cudaError_t launch_dh_pair(const ChunkParams& p, const CUtensorMap& mDS, const CUtensorMap& mWmn, int n_sm,
                           bool bf16, bool wide, cudaStream_t st);
cudaError_t launch_dw_pair(const ChunkParams& p, const CUtensorMap& mDSmn, const CUtensorMap& mHcmn, int n_sm,
                           bool bf16, cudaStream_t st);
cudaError_t launch_dh_pair_fp8(const ChunkParams& p, const CUtensorMap& mQa, const CUtensorMap& mWmn, int n_sm,
                               bool wide, cudaStream_t st);
cudaError_t launch_dw_pair_fp8(const ChunkParams& p, const CUtensorMap& mQbmn, const CUtensorMap& mHqmn, int n_sm,
                               cudaStream_t st);

}  // namespace grpo
