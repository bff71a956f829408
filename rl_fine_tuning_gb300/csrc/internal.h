// Host/device declarations shared by the translation units of libgrpo.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "grpo.h"

namespace grpo {

constexpr int kBM = 128;              // rows (or vocabulary rows for dW) per MMA tile
constexpr int kBK = 64;               // K elements per pipeline stage: one 128-byte swizzle span
constexpr int kBN = 256;              // accumulator columns per MMA tile
constexpr int kMaxFwdSplits = 8;      // vocabulary splits of one forward row tile
constexpr int kDefaultChunkRows = 8192;
constexpr int kMergeThreads = 256;
constexpr int kIndexThreads = 1024;
// CTAs per cluster sharing one B tile through TMA multicast (1, 2 or 4)
constexpr int kClusterFwd = 2;
constexpr int kClusterBwd = 2;

// int32 words at the start of the workspace
enum CountSlot {
    C_NVALID = 0,      // masked-in rows
    C_NTILES = 1,      // forward row tiles
    C_NCHUNKS = 2,     // backward chunks
    C_CHUNK_ROWS = 3,  // rows per backward chunk (multiple of 128)
    C_WINV = 4,        // 1 / max(N_valid, 1) as float bits
    C_COUNT_WORDS = 16
};

struct WsLayout {
    size_t counts, tiles, rows, part, zt, lse, gco, blocksum, hc, ds, total;
    int S;           // forward vocabulary splits
    int nps;         // vocabulary N-tiles per split
    int n_ntiles;    // ceil(V / kBN)
    int R;           // rows per backward chunk (buffer height)
    int V_pad;       // row pitch of the dlogits buffer, elements
    int nblk;        // merge blocks
    int64_t N;
};

bool ws_layout(const grpo_shape& s, WsLayout* out);

struct FwdParams {
    const int2* tiles;      // (first row, rows) per forward tile
    const int* counts;
    const int* tokens;
    float4* part;           // [N x S] (m_pol, s_pol, m_ref, s_ref)
    float2* zt;             // [N] (z_pol[tok], z_ref[tok])
    int64_t N;
    int V, d, S, nps, n_ntiles;
    int* status;
};

struct ChunkParams {
    const int* counts;
    const int* rows;        // valid-row list
    const int* tokens;
    const float* lse;       // [N] policy logsumexp
    const float* gco;       // [N] d ell / d q
    float scale;            // loss scale
    int chunk;
    int V, d, V_pad;
    uint16_t* dS;           // [R x V_pad] scaled dlogits (without the 1/N_valid factor)
    uint16_t* dH;           // [N x d]
    float* dW;              // [V x d]
    int* found_inf;
    int* status;
};

// ---- launches (return cudaError_t of the launch) ----
cudaError_t launch_index(const uint8_t* mask, int64_t N, int R_max, int* counts, int* rows, int2* tiles,
                         int* status, int* found_inf, cudaStream_t st);
cudaError_t launch_advantages(const float* r, int n_groups, int G, float eps, int std_unbiased, float* adv,
                              cudaStream_t st);
cudaError_t launch_build_mask(const int32_t* lengths, int n_seq, int L, uint8_t* mask, cudaStream_t st);
cudaError_t launch_merge(const WsLayout& ws, char* wsp, const uint8_t* mask, const int* tokens,
                         const float* adv, int L, int V, float beta, float* loss_out, float* row_stats,
                         int* status, cudaStream_t st);
cudaError_t launch_gather_rows(const ChunkParams& p, const void* h_pol, void* hc, int R, cudaStream_t st);
cudaError_t launch_clear_grads(const int* counts, int* found_inf, float* dW, int64_t n, cudaStream_t st);
cudaError_t launch_zero_masked_rows(const uint8_t* mask, int64_t N, int d, void* dH, cudaStream_t st);

cudaError_t launch_fwd(const FwdParams& p, const CUtensorMap& mHp, const CUtensorMap& mHr,
                       const CUtensorMap& mW, int n_sm, bool bf16, cudaStream_t st);
cudaError_t launch_ds(const ChunkParams& p, const CUtensorMap& mHc, const CUtensorMap& mW, int n_sm, bool bf16,
                      cudaStream_t st);
cudaError_t launch_dh(const ChunkParams& p, const CUtensorMap& mDS, const CUtensorMap& mWmn, int n_sm,
                      bool bf16, cudaStream_t st);
cudaError_t launch_dw(const ChunkParams& p, const CUtensorMap& mDSmn, const CUtensorMap& mHcmn, int n_sm,
                      bool bf16, cudaStream_t st);

}  // namespace grpo
