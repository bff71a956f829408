// The steps of the GRPO loss that are not GEMMs: advantages, mask / row
// index, logsumexp merge + objective + deterministic loss, row gather, the
// dlogits pass over the kept exponentials (HBM-bound), zeroing, and the
// self-test of the checked build.
#include <cfloat>
#include <cmath>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"

namespace grpo {

// ------------------------------------------------------------ advantages
// Group-relative advantage, fp64 with a fixed summation order and explicit
// round-to-nearest operations (no contraction), so the result is the same
// bit pattern on every run ("Train your own R1 reasoning model with Unsloth",
// section 3: score, group mean, compare each score with it).
__global__ void k_advantages(const float* __restrict__ r, int n_groups, int G, float eps, int std_unbiased,
                             float* __restrict__ adv) {
    const int gi = blockIdx.x * blockDim.x + threadIdx.x;
    if (gi >= n_groups) return;
    const float* rr = r + static_cast<size_t>(gi) * G;
    double sum = 0.0;
    for (int i = 0; i < G; ++i) sum = __dadd_rn(sum, static_cast<double>(rr[i]));
    const double mu = __ddiv_rn(sum, static_cast<double>(G));
    double ss = 0.0;
    for (int i = 0; i < G; ++i) {
        const double dv = __dsub_rn(static_cast<double>(rr[i]), mu);
        ss = __dadd_rn(ss, __dmul_rn(dv, dv));
    }
    const int div = std_unbiased ? G - 1 : G;
    const double sigma = div > 0 ? __dsqrt_rn(__ddiv_rn(ss, static_cast<double>(div))) : 0.0;
    const double den = __dadd_rn(sigma, static_cast<double>(eps));
    for (int i = 0; i < G; ++i)
        adv[static_cast<size_t>(gi) * G + i] =
            __double2float_rn(__ddiv_rn(__dsub_rn(static_cast<double>(rr[i]), mu), den));
}

cudaError_t launch_advantages(const float* r, int n_groups, int G, float eps, int std_unbiased, float* adv,
                              cudaStream_t st) {
    const int thr = 128;
    k_advantages<<<(n_groups + thr - 1) / thr, thr, 0, st>>>(r, n_groups, G, eps, std_unbiased, adv);
    return cudaGetLastError();
}

// ------------------------------------------------------------ mask
__global__ void k_build_mask(const int32_t* __restrict__ lengths, int n_seq, int L, uint8_t* __restrict__ mask) {
    const int64_t n = static_cast<int64_t>(n_seq) * L;
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < n;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int i = static_cast<int>(t / L);
        const int j = static_cast<int>(t - static_cast<int64_t>(i) * L);
        mask[t] = static_cast<uint8_t>(j < lengths[i]);
    }
}

cudaError_t launch_build_mask(const int32_t* lengths, int n_seq, int L, uint8_t* mask, cudaStream_t st) {
    const int64_t n = static_cast<int64_t>(n_seq) * L;
    int blocks = static_cast<int>((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    k_build_mask<<<blocks, 256, 0, st>>>(lengths, n_seq, L, mask);
    return cudaGetLastError();
}

// ------------------------------------------------------------ row index
// One block walks the mask in segments of kIndexThreads*kItems rows, carrying
// the running counts between segments.  Outputs, all in ascending row order:
//   rows[]  -- every masked-in row
//   tiles[] -- forward row tiles: runs of consecutive masked-in rows cut into
//              pieces of at most kBM rows (first row, row count)
// and the chunking of the backward pass over the valid-row list.
constexpr int kItems = 16;

__device__ __forceinline__ int block_excl_sum(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[w] = x;
    __syncthreads();
    if (w == 0) {
        int y = lane < nw ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int z = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += z;
        }
        if (lane < nw) s_warp[lane] = y;
    }
    __syncthreads();
    const int off = w > 0 ? s_warp[w - 1] : 0;
    *total = s_warp[nw - 1];
    __syncthreads();
    return off + x - v;
}

__device__ __forceinline__ int block_excl_max(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x = max(x, y);
    }
    int excl_in_warp = __shfl_up_sync(0xffffffffu, x, 1);
    if (lane == 0) excl_in_warp = -1;
    if (lane == 31) s_warp[w] = x;
    __syncthreads();
    if (w == 0) {
        int y = lane < nw ? s_warp[lane] : -1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int z = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y = max(y, z);
        }
        if (lane < nw) s_warp[lane] = y;
    }
    __syncthreads();
    const int off = w > 0 ? s_warp[w - 1] : -1;
    *total = s_warp[nw - 1];
    __syncthreads();
    return max(off, excl_in_warp);
}

__global__ void __launch_bounds__(kIndexThreads) k_index(const uint8_t* __restrict__ mask, int64_t N, int R_max,
                                                         int* __restrict__ counts, int* __restrict__ rows,
                                                         int2* __restrict__ tiles, int* __restrict__ sched,
                                                         int n_sched, int* status) {
    __shared__ int s_warp[32];
    const int tid = threadIdx.x;
    if (tid == 0) *status = 0;
    for (int i = tid; i < n_sched; i += kIndexThreads) sched[i] = 0;
    int carry_valid = 0, carry_tiles = 0, carry_lastzero = -1;
    for (int64_t base = 0; base < N; base += static_cast<int64_t>(kIndexThreads) * kItems) {
        const int t0 = static_cast<int>(base) + tid * kItems;
        uint32_t bits = 0;
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
            const int64_t t = static_cast<int64_t>(t0) + k;
            if (t < N && mask[t] != 0) bits |= 1u << k;
        }
        int nv = __popc(bits);
        int lz = -1;
#pragma unroll
        for (int k = 0; k < kItems; ++k)
            if (!((bits >> k) & 1u)) lz = t0 + k;
        int tot_nv, tot_lz, tot_ns;
        const int nv_excl = block_excl_sum(nv, s_warp, &tot_nv);
        const int lz_excl = block_excl_max(lz, s_warp, &tot_lz);
        const int last_zero = max(carry_lastzero, lz_excl);
        int ns = 0;
        {
            int lzr = last_zero;
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
                if (!((bits >> k) & 1u)) {
                    lzr = t0 + k;
                } else if ((((t0 + k) - lzr - 1) & (kBM - 1)) == 0) {
                    ++ns;
                }
            }
        }
        const int ns_excl = block_excl_sum(ns, s_warp, &tot_ns);
        {
            int vi = carry_valid + nv_excl, ti = carry_tiles + ns_excl, lzr = last_zero;
#pragma unroll
            for (int k = 0; k < kItems; ++k) {
                const int t = t0 + k;
                if (!((bits >> k) & 1u)) {
                    lzr = t;
                } else {
                    if (GRPO_DCHECK(vi < N, status)) rows[vi] = t;
                    ++vi;
                    if (((t - lzr - 1) & (kBM - 1)) == 0) {
                        if (GRPO_DCHECK(ti < N, status)) tiles[ti] = make_int2(t, 0);
                        ++ti;
                    }
                }
            }
        }
        carry_valid += tot_nv;
        carry_tiles += tot_ns;
        carry_lastzero = max(carry_lastzero, tot_lz);
    }
    if (tid == 0) {
        const int nv = carry_valid;
        // fixed-size chunks of R_max rows (a multiple of kBM); the last one holds the rest
        const int n_chunks = nv > 0 ? (nv + R_max - 1) / R_max : 0;
        const int rc = n_chunks > 0 ? R_max : 0;
        counts[C_NVALID] = nv;
        counts[C_NTILES] = carry_tiles;
        counts[C_NCHUNKS] = n_chunks;
        counts[C_CHUNK_ROWS] = rc;
        counts[C_WINV] = __float_as_int(1.0f / static_cast<float>(nv > 0 ? nv : 1));
        counts[C_NACT] = 0;   // counted by k_seq_counts
        counts[C_SHARD] = 0;  // set by k_apply_global_counts for a shard
        counts[C_NDIV_G] = 0;
        counts[C_NACT_G] = 0;
    }
}

// rows covered by each forward tile: up to kBM, stopping at the end of the run
__global__ void k_tile_rows(const uint8_t* __restrict__ mask, int64_t N, const int* __restrict__ counts,
                            int2* __restrict__ tiles) {
    const int n_tiles = counts[C_NTILES];
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_tiles; i += gridDim.x * blockDim.x) {
        const int t0 = tiles[i].x;
        int n = 1;
        while (n < kBM && static_cast<int64_t>(t0) + n < N && mask[t0 + n] != 0) ++n;
        tiles[i].y = n;
    }
}

cudaError_t launch_index(const uint8_t* mask, int64_t N, int R_max, int* counts, int* rows, int2* tiles,
                         int* sched, int n_sched, int* status, cudaStream_t st) {
    k_index<<<1, kIndexThreads, 0, st>>>(mask, N, R_max, counts, rows, tiles, sched, n_sched, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int blocks = static_cast<int>((N / kBM + 255) / 256) + 1;
    if (blocks > 1024) blocks = 1024;
    k_tile_rows<<<blocks, 256, 0, st>>>(mask, N, counts, tiles);
    return cudaGetLastError();
}

// ------------------------------------------------------------ merge + objective
// The split partials of one row, part[0 .. S), merged by one warp: lane k
// takes splits k, k+32, ...; the maxima and then the rescaled sums are
// combined across the warp in a fixed butterfly order.  Lane 0's results are
// the ones used (every lane combines in its own order).
__device__ __forceinline__ void merge_lse_warp(const float4* __restrict__ part, int S, int lane, float* lse_pol,
                                               float* lse_ref, float* max_pol) {
    float mp = -INFINITY, mr = -INFINITY;
    for (int k = lane; k < S; k += 32) {
        const float4 ps = part[k];
        mp = fmaxf(mp, ps.x);
        mr = fmaxf(mr, ps.z);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, o));
        mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, o));
    }
    float sp = 0.f, sr = 0.f;
    for (int k = lane; k < S; k += 32) {
        const float4 ps = part[k];
        sp += ps.y * expf(ps.x - mp);
        sr += ps.w * expf(ps.z - mr);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sp += __shfl_xor_sync(0xffffffffu, sp, o);
        sr += __shfl_xor_sync(0xffffffffu, sr, o);
    }
    *lse_pol = mp + logf(sp);
    *lse_ref = mr + logf(sr);
    *max_pol = mp;
}

// Per row: merge the per-split (max, sum-exp) partials of the policy and the
// reference logits into their logsumexp, form q, p, the reverse-KL term
// exp(p-q) - (p-q) - 1 = expm1(x) - x, the per-token objective and its
// derivative w.r.t. q ("Long-context GRPO", section 4).  The masked sum of the
// objective is reduced in fp64 along a fixed tree afterwards.
// One warp per row: all rows t in [0, N) (chunk < 0), or the valid rows of
// one backward chunk.  Writes lse_pol, g = d ell / d q and ell per row.
__global__ void __launch_bounds__(kMergeThreads) k_merge(const MergeParams p) {
    const int64_t row = (blockIdx.x * static_cast<int64_t>(kMergeThreads) + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    int64_t t, pidx;
    if (p.chunk < 0) {
        t = row;
        if (t >= p.N) return;
        pidx = t;
    } else {
        if (p.chunk >= p.counts[C_NCHUNKS]) return;
        const int rc = p.counts[C_CHUNK_ROWS];
        const int c0 = p.chunk * rc;
        const int n_c = min(rc, p.counts[C_NVALID] - c0);
        if (row >= n_c || !GRPO_DCHECK(row < p.R, p.status)) return;
        t = p.rows[c0 + row];
        pidx = row;
        if (!GRPO_DCHECK(t >= 0 && t < p.N, p.status)) return;   // uniform across the warp
    }
    // t is uniform across the warp from here on
    float lse_p = 0.f, lse_r = 0.f, q = 0.f, p_ = 0.f, pen = 0.f, g = 0.f, ell = 0.f, zmax = 0.f;
    if (p.mask[t]) {
        const int tok = p.tokens[t];
        if (tok < 0 || tok >= p.V) {
            if (lane == 0) atomicCAS(p.status, 0, GRPO_ERR_SHAPE);
        } else {
            merge_lse_warp(p.part + pidx * p.S, p.S, lane, &lse_p, &lse_r, &zmax);
            const float2 z = p.zt[t];
            q = z.x - lse_p;
            p_ = z.y - lse_r;
            const float x = p_ - q;
            const float A = p.adv[t / p.L];
            // penalty and d ell / d q of the chosen objective (x = p - q)
            switch (p.objective) {
                case GRPO_OBJ_NO_DETACH: {
                    const float em1 = expm1f(x);
                    pen = em1 - x;
                    g = -p.beta * em1;   // exp(q - q) is constant: no policy-gradient term
                    break;
                }
                case GRPO_OBJ_REVERSE_KL_Q: {
                    const float eq = expf(q);
                    pen = eq * (expm1f(x) - x);
                    g = -A - p.beta * x * eq;
                    break;
                }
                case GRPO_OBJ_FORWARD_KL: {
                    const float em1n = expm1f(-x);
                    pen = em1n + x;
                    g = -A + p.beta * em1n;
                    break;
                }
                default: {
                    const float em1 = expm1f(x);
                    pen = em1 - x;
                    g = -A - p.beta * em1;
                    break;
                }
            }
            ell = -A + p.beta * pen;
            if (p.loss_mode == GRPO_SEQUENCE_MEAN) {
                // weight N_v / (n_active * len_i): the final division by N_v
                // then yields the mean over completions of their token means
                // (for a shard, N_v and n_active count every shard's rows)
                const int nv = count_ndiv(p.counts);
                const int nact = count_nact(p.counts);
                const int len = p.seqcnt[t / p.L];
                const float rel = static_cast<float>(static_cast<double>(nv) /
                                                     (static_cast<double>(nact) * static_cast<double>(len)));
                ell *= rel;
                g *= rel;
            }
        }
    }
    if (lane != 0) return;
    p.lse[t] = lse_p;
    p.gco[t] = g;
    p.ell[t] = ell;
    if (p.rmax) p.rmax[t] = zmax;
    if (p.row_stats) {
        float* o = p.row_stats + t * 5;
        o[0] = lse_p;
        o[1] = lse_r;
        o[2] = q;
        o[3] = p_;
        o[4] = pen;
    }
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t st) {
    const int64_t n = p.chunk < 0 ? p.N : static_cast<int64_t>(p.R);   // rows, one warp each
    constexpr int kRowsPerBlock = kMergeThreads / 32;
    int64_t blocks = (n + kRowsPerBlock - 1) / kRowsPerBlock;
    if (blocks < 1) blocks = 1;
    k_merge<<<static_cast<unsigned>(blocks), kMergeThreads, 0, st>>>(p);
    return cudaGetLastError();
}

// masked-in rows per completion; completions with any count toward C_NACT
__global__ void k_seq_counts(const uint8_t* __restrict__ mask, int n_seq, int L, int* __restrict__ seqcnt,
                             int* __restrict__ counts) {
    __shared__ int sh[256];
    for (int i = blockIdx.x; i < n_seq; i += gridDim.x) {
        const uint8_t* m = mask + static_cast<int64_t>(i) * L;
        int c = 0;
        for (int j = threadIdx.x; j < L; j += 256) c += m[j] != 0;
        sh[threadIdx.x] = c;
        __syncthreads();
        for (int s = 128; s > 0; s >>= 1) {
            if (threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            seqcnt[i] = sh[0];
            if (sh[0] > 0) atomicAdd(counts + C_NACT, 1);
        }
        __syncthreads();
    }
}

cudaError_t launch_seq_counts(const uint8_t* mask, int n_seq, int L, int* seqcnt, int* counts, cudaStream_t st) {
    int blocks = n_seq < 4096 ? n_seq : 4096;
    if (blocks < 1) blocks = 1;
    k_seq_counts<<<blocks, 256, 0, st>>>(mask, n_seq, L, seqcnt, counts);
    return cudaGetLastError();
}

// ------------------------------------------------------------ data-parallel shards
// One shard's counts: out[0] = masked-in rows, out[1] = completions with at
// least one masked-in row (out zeroed beforehand; integer atomics, so the
// result does not depend on the order the blocks finish in).
__global__ void k_shard_counts(const uint8_t* __restrict__ mask, int n_seq, int L, int* __restrict__ out) {
    __shared__ int sh[256];
    for (int i = blockIdx.x; i < n_seq; i += gridDim.x) {
        const uint8_t* m = mask + static_cast<int64_t>(i) * L;
        int c = 0;
        for (int j = threadIdx.x; j < L; j += 256) c += m[j] != 0;
        sh[threadIdx.x] = c;
        __syncthreads();
        for (int s = 128; s > 0; s >>= 1) {
            if (threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
            __syncthreads();
        }
        if (threadIdx.x == 0 && sh[0] > 0) {
            atomicAdd(out, sh[0]);
            atomicAdd(out + 1, 1);
        }
        __syncthreads();
    }
}

cudaError_t launch_shard_counts(const uint8_t* mask, int n_seq, int L, int* out, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(out, 0, 2 * sizeof(int), st);
    if (e != cudaSuccess) return e;
    int blocks = n_seq < 4096 ? n_seq : 4096;
    if (blocks < 1) blocks = 1;
    k_shard_counts<<<blocks, 256, 0, st>>>(mask, n_seq, L, out);
    return cudaGetLastError();
}

// A shard of a data-parallel batch ("partition by whole prompt groups"): the
// token mean divides by the masked-in rows of ALL shards, and the sequence
// mean by all shards' active completions, so the shards' losses and dW add up
// to those of the whole batch.  Runs after the row index (and the completion
// counts): global counts smaller than this shard's own are an error.
__global__ void k_apply_global_counts(const int* __restrict__ g, int* __restrict__ counts, int loss_mode,
                                      int* status) {
    const int nv_g = g[0], nact_g = g[1];
    const bool bad = nv_g < counts[C_NVALID] || (loss_mode == GRPO_SEQUENCE_MEAN && nact_g < counts[C_NACT]);
    if (bad) atomicCAS(status, 0, GRPO_ERR_SHAPE);
    counts[C_SHARD] = 1;
    counts[C_NDIV_G] = nv_g;
    counts[C_NACT_G] = nact_g;
    counts[C_WINV] = __float_as_int(1.0f / static_cast<float>(nv_g > 0 ? nv_g : 1));
}

cudaError_t launch_apply_global_counts(const int* global_counts, int* counts, int loss_mode, int* status,
                                       cudaStream_t st) {
    k_apply_global_counts<<<1, 1, 0, st>>>(global_counts, counts, loss_mode, status);
    return cudaGetLastError();
}

// masked rows: objective 0 and zero diagnostics (the chunked merge never visits them)
__global__ void k_rows_init(const uint8_t* __restrict__ mask, int64_t N, float* __restrict__ ell,
                            float* __restrict__ row_stats) {
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < N;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        if (mask[t]) continue;
        ell[t] = 0.f;
        if (row_stats)
            for (int j = 0; j < 5; ++j) row_stats[t * 5 + j] = 0.f;
    }
}

cudaError_t launch_rows_init(const uint8_t* mask, int64_t N, float* ell, float* row_stats, int sm_count,
                             cudaStream_t st) {
    int blocks = static_cast<int>((N + 255) / 256);
    if (blocks > sm_count * 8) blocks = sm_count * 8;
    if (blocks < 1) blocks = 1;
    k_rows_init<<<blocks, 256, 0, st>>>(mask, N, ell, row_stats);
    return cudaGetLastError();
}

// Masked mean of the per-row objective: fp64 sums over fixed blocks of rows in
// a fixed tree, then one block sums the block results in a fixed order.
__global__ void __launch_bounds__(kMergeThreads) k_loss_blocks(const float* __restrict__ ell, int64_t N,
                                                               double* __restrict__ blocksum) {
    __shared__ double sh[kMergeThreads];
    const int64_t t = blockIdx.x * static_cast<int64_t>(kMergeThreads) + threadIdx.x;
    sh[threadIdx.x] = t < N ? static_cast<double>(ell[t]) : 0.0;
    __syncthreads();
#pragma unroll
    for (int s = kMergeThreads / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) blocksum[blockIdx.x] = sh[0];
}

__global__ void __launch_bounds__(1024) k_loss_final(const double* __restrict__ blocksum, int nblk,
                                                     const int* __restrict__ counts, float* __restrict__ loss_out) {
    __shared__ double sh[1024];
    double acc = 0.0;
    for (int i = threadIdx.x; i < nblk; i += 1024) acc += blocksum[i];
    sh[threadIdx.x] = acc;
    __syncthreads();
    for (int s = 512; s > 0; s >>= 1) {
        if (threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const int nv = count_ndiv(counts);
        *loss_out = nv > 0 ? static_cast<float>(sh[0] / static_cast<double>(nv)) : 0.f;
    }
}

cudaError_t launch_loss_reduce(const float* ell, int64_t N, double* blocksum, int nblk, const int* counts,
                               float* loss_out, cudaStream_t st) {
    k_loss_blocks<<<nblk, kMergeThreads, 0, st>>>(ell, N, blocksum);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_loss_final<<<1, 1024, 0, st>>>(blocksum, nblk, counts, loss_out);
    return cudaGetLastError();
}

// ------------------------------------------------------------ gather / zero
// Hc[slot] = h_pol[rows[c0 + slot]] (and Hcr from h_ref when given) for the
// chunk's slots; the slots after the last one, up to the next multiple of kBM,
// are zeroed.
__global__ void k_gather_rows(const int* __restrict__ counts, const int* __restrict__ rows, int chunk,
                              const uint4* __restrict__ h, uint4* __restrict__ hc, const uint4* __restrict__ hr,
                              uint4* __restrict__ hcr, int vec_per_row, int R, int64_t N, int* status) {
    if (chunk >= counts[C_NCHUNKS]) return;
    const int rc = counts[C_CHUNK_ROWS];
    const int c0 = chunk * rc;
    const int n_c = min(rc, counts[C_NVALID] - c0);
    const int n_fill = min(R, (n_c + kBM - 1) / kBM * kBM);
    const int64_t total = static_cast<int64_t>(n_fill) * vec_per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int slot = static_cast<int>(i / vec_per_row);
        const int v = static_cast<int>(i - static_cast<int64_t>(slot) * vec_per_row);
        uint4 x = make_uint4(0, 0, 0, 0), y = make_uint4(0, 0, 0, 0);
        if (slot < n_c && GRPO_DCHECK(rows[c0 + slot] >= 0 && rows[c0 + slot] < N, status)) {
            const int64_t src = static_cast<int64_t>(rows[c0 + slot]) * vec_per_row + v;
            x = h[src];
            if (hr) y = hr[src];
        }
        hc[i] = x;
        if (hcr) hcr[i] = y;
    }
}

// The gather of 16-bit rows, one 64-row x 64-column tile per block iteration:
// hc and hcr as above, and hct[k][slot] = hc[slot][k] ([d x R], pitch R) through
// a shared-memory tile of 32-bit words (two columns each; 33 words per row, so
// the column reads of the transposed write hit distinct banks up to 2-way).
constexpr int kGatherTile = 64;

__global__ void __launch_bounds__(256) k_gather_rows_t(const int* __restrict__ counts, const int* __restrict__ rows,
                                                       int chunk, const uint4* __restrict__ h, uint4* __restrict__ hc,
                                                       const uint4* __restrict__ hr, uint4* __restrict__ hcr,
                                                       uint16_t* __restrict__ hct, int d, int R, int64_t N,
                                                       int* status) {
    __shared__ uint32_t tile[kGatherTile][kGatherTile / 2 + 1];
    if (chunk >= counts[C_NCHUNKS]) return;
    const int rc = counts[C_CHUNK_ROWS];
    const int c0 = chunk * rc;
    const int n_c = min(rc, counts[C_NVALID] - c0);
    const int n_fill = min(R, (n_c + kBM - 1) / kBM * kBM);   // a multiple of 128
    const int nt_d = d / kGatherTile;
    const int n_tiles = (n_fill / kGatherTile) * nt_d;
    const int vpr = d / 8;                                    // 16-byte vectors per row
    for (int tix = blockIdx.x; tix < n_tiles; tix += gridDim.x) {
        const int r0 = (tix / nt_d) * kGatherTile;
        const int d0 = (tix % nt_d) * kGatherTile;
        for (int i = threadIdx.x; i < kGatherTile * 8; i += blockDim.x) {
            const int r = i >> 3, v = i & 7;
            const int slot = r0 + r;
            uint4 x = make_uint4(0, 0, 0, 0), y = make_uint4(0, 0, 0, 0);
            if (slot < n_c) {
                const int t = rows[c0 + slot];
                if (GRPO_DCHECK(t >= 0 && t < N, status)) {
                    const int64_t src = static_cast<int64_t>(t) * vpr + (d0 >> 3) + v;
                    x = h[src];
                    y = hr[src];
                }
            }
            const int64_t dst = static_cast<int64_t>(slot) * vpr + (d0 >> 3) + v;
            hc[dst] = x;
            hcr[dst] = y;
            tile[r][4 * v] = x.x;
            tile[r][4 * v + 1] = x.y;
            tile[r][4 * v + 2] = x.z;
            tile[r][4 * v + 3] = x.w;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kGatherTile * 8; i += blockDim.x) {
            const int k = i >> 3, v = i & 7;   // output row d0 + k, slots r0 + 8v .. r0 + 8v + 7
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t w0 = tile[8 * v + 2 * j][k >> 1], w1 = tile[8 * v + 2 * j + 1][k >> 1];
                const uint32_t e0 = (k & 1) ? (w0 >> 16) : (w0 & 0xFFFFu);
                const uint32_t e1 = (k & 1) ? (w1 >> 16) : (w1 & 0xFFFFu);
                o[j] = e0 | (e1 << 16);
            }
            *reinterpret_cast<uint4*>(hct + static_cast<int64_t>(d0 + k) * R + r0 + 8 * v) =
                make_uint4(o[0], o[1], o[2], o[3]);
        }
        __syncthreads();
    }
}

cudaError_t launch_gather_rows_t(const ChunkParams& p, const void* h_pol, void* hc, const void* h_ref, void* hcr,
                                 void* hct, int R, int sm_count, cudaStream_t st) {
    const int64_t tiles = static_cast<int64_t>(R / kGatherTile) * (p.d / kGatherTile);
    int blocks = static_cast<int>(tiles < sm_count * 8 ? tiles : sm_count * 8);
    if (blocks < 1) blocks = 1;
    k_gather_rows_t<<<blocks, 256, 0, st>>>(p.counts, p.rows, p.chunk, static_cast<const uint4*>(h_pol),
                                            static_cast<uint4*>(hc), static_cast<const uint4*>(h_ref),
                                            static_cast<uint4*>(hcr), static_cast<uint16_t*>(hct), p.d, R, p.N,
                                            p.status);
    return cudaGetLastError();
}

#ifdef GRPO_DEVICE_CHECKS
// One thread stores one past the end of a 16-element shared array through the
// checked access pattern of the kernels: the check refuses the store and
// records GRPO_ERR_BOUNDS.  Exists only in the checked build.
__global__ void k_bounds_selftest(int* status) {
    __shared__ int buf[16];
    *status = 0;
    const int i = 16 + static_cast<int>(threadIdx.x);
    if (GRPO_DCHECK(i < 16, status)) buf[i] = 1;
}

cudaError_t launch_bounds_selftest(int* status, cudaStream_t st) {
    k_bounds_selftest<<<1, 1, 0, st>>>(status);
    return cudaGetLastError();
}
#endif

cudaError_t launch_gather_rows(const ChunkParams& p, const void* h_pol, void* hc, const void* h_ref, void* hcr, int R,
                               int row_bytes, int sm_count, cudaStream_t st) {
    const int vpr = row_bytes / 16;
    const int64_t total = static_cast<int64_t>(R) * vpr;
    int blocks = static_cast<int>((total + 255) / 256);
    if (blocks > sm_count * 16) blocks = sm_count * 16;
    k_gather_rows<<<blocks, 256, 0, st>>>(p.counts, p.rows, p.chunk, static_cast<const uint4*>(h_pol),
                                          static_cast<uint4*>(hc), static_cast<const uint4*>(h_ref),
                                          static_cast<uint4*>(hcr), vpr, R, p.N, p.status);
    return cudaGetLastError();
}

// ------------------------------------------------------------ dlogits from stored exponentials
// In place over the chunk buffer: the forward left e = exp(z - m) (bf16) for
// every policy logit and m, the running max after each 32-column group.  With
// the row's logsumexp the softmax is p = e * exp(m - lse), and
//   dS = s * g * (onehot(tok) - p)
// is written back in the storage dtype.  The sampled token's entry uses
// p_tok = exp(z[tok] - lse) in fp32, so 1 - p_tok keeps full precision.
// Slots past the chunk's last row (to the next multiple of kBM) become 0.
template <bool kBf16>
__global__ void __launch_bounds__(kTransformThreads) k_transform(const ChunkParams p, int R) {
    if (p.chunk >= p.counts[C_NCHUNKS]) return;
    const int rc = p.counts[C_CHUNK_ROWS];
    const int c0 = p.chunk * rc;
    const int n_c = min(rc, p.counts[C_NVALID] - c0);
    const int n_fill = min(R, (n_c + kBM - 1) / kBM * kBM);
    const int nvec = (p.V + 7) / 8;   // 8 elements (16 bytes) per vector; V_pad is a multiple of 64
    bool bad = false;
    for (int slot = blockIdx.x; slot < n_fill; slot += gridDim.x) {
        uint4* row = reinterpret_cast<uint4*>(p.dS + static_cast<int64_t>(slot) * p.V_pad);
        if (slot >= n_c) {
            for (int i = threadIdx.x; i < nvec; i += kTransformThreads) row[i] = make_uint4(0, 0, 0, 0);
            continue;
        }
        const int t = p.rows[c0 + slot];
        if (!GRPO_DCHECK(t >= 0 && t < p.N, p.status)) continue;
        const int tok = p.tokens[t];
        const float lse = p.lse[t];
        const float coef = p.scale * p.gco[t];
        const float ptok = expf(p.zt[t].x - lse);
        const float* mrow = p.mx + static_cast<int64_t>(slot) * p.nc32;
        for (int i = threadIdx.x; i < nvec; i += kTransformThreads) {
            const int v0 = i * 8;
            const float c = coef * expf(mrow[v0 >> 5] - lse);
            uint4 u = row[i];
            uint32_t w[4] = {u.x, u.y, u.z, u.w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float e0 = __uint_as_float(w[j] << 16);
                const float e1 = __uint_as_float(w[j] & 0xFFFF0000u);
                const int va = v0 + 2 * j, vb = va + 1;
                float d0 = -c * e0, d1 = -c * e1;
                if (va == tok) d0 = coef * (1.f - ptok);
                if (vb == tok) d1 = coef * (1.f - ptok);
                if (va >= p.V) d0 = 0.f;
                if (vb >= p.V) d1 = 0.f;
                uint16_t h0, h1;
                if (kBf16) {
                    h0 = __bfloat16_as_ushort(__float2bfloat16_rn(d0));
                    h1 = __bfloat16_as_ushort(__float2bfloat16_rn(d1));
                } else {
                    h0 = __half_as_ushort(__float2half_rn(d0));
                    h1 = __half_as_ushort(__float2half_rn(d1));
                    bad |= ((h0 & 0x7C00u) == 0x7C00u) || ((h1 & 0x7C00u) == 0x7C00u);
                }
                o[j] = static_cast<uint32_t>(h0) | (static_cast<uint32_t>(h1) << 16);
            }
            row[i] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    if (!kBf16 && __syncthreads_or(bad) && threadIdx.x == 0) atomicOr(p.found_inf, 1);
}

cudaError_t launch_transform(const ChunkParams& p, bool bf16, int R, int sm_count, cudaStream_t st) {
    int blocks = R;
    if (blocks > sm_count * 8) blocks = sm_count * 8;
    if (bf16)
        k_transform<true><<<blocks, kTransformThreads, 0, st>>>(p, R);
    else
        k_transform<false><<<blocks, kTransformThreads, 0, st>>>(p, R);
    return cudaGetLastError();
}

// ------------------------------------------------------------ 8-bit backward
// The dlogits of a row are dS = g (onehot(tok) - softmax).  The 8-bit backward
// keeps the one-hot part exact (the GEMM epilogues add it) and sends only
// P = g * softmax through 8-bit codes.  |P| <= |g| exp(m_grp - lse) for every
// column of a 32-column group whose running max is m_grp, and the row's
// largest |P| is |g| exp(max z - lse).

// gmax[grp] = max over the chunk's rows of |g| exp(m_grp - lse): one bound of
// |P| per 32-column group, shared by all rows of the chunk (zeroed
// beforehand; non-negative floats order like their bit patterns).  A block
// takes kF8GroupRows rows and keeps max_t (m_grp + log|g_t| - lse_t) per group,
// so it needs one exponential per group; rows with g = 0 add nothing.
constexpr int kF8GroupRows = 16;

__global__ void __launch_bounds__(256) k_f8_group_max(const ChunkParams p) {
    __shared__ float c_row[kF8GroupRows];
    if (p.chunk >= p.counts[C_NCHUNKS]) return;
    const int rc = p.counts[C_CHUNK_ROWS];
    const int c0 = p.chunk * rc;
    const int n_c = min(rc, p.counts[C_NVALID] - c0);
    const int s0 = blockIdx.x * kF8GroupRows;
    if (s0 >= n_c) return;
    const int nr = min(n_c - s0, kF8GroupRows);
    if (threadIdx.x < kF8GroupRows) {
        float c = -INFINITY;
        const int slot = s0 + threadIdx.x;
        if (static_cast<int>(threadIdx.x) < nr) {
            const int t = p.rows[c0 + slot];
            if (GRPO_DCHECK(t >= 0 && t < p.N && slot < p.R, p.status)) {
                const float g = fabsf(p.gco[t]);
                c = g > 0.f ? logf(g) - p.lse[t] : -INFINITY;
            }
            // tokpos[tok] = index of the token's first key in the chunk's sorted keys
            const uint32_t tok = static_cast<uint32_t>(p.keys[slot] >> 32);
            if ((slot == 0 || static_cast<uint32_t>(p.keys[slot - 1] >> 32) != tok) && tok < static_cast<uint32_t>(p.V))
                p.tokpos[tok] = slot;
        }
        c_row[threadIdx.x] = c;
    }
    __syncthreads();
    const int ng = (p.V + 31) / 32;
    const float* mx0 = p.mx + static_cast<int64_t>(s0) * p.nc32;
    for (int grp = threadIdx.x; grp < ng; grp += blockDim.x) {
        float m = -INFINITY;
#pragma unroll
        for (int r = 0; r < kF8GroupRows; ++r)
            if (r < nr) m = fmaxf(m, mx0[static_cast<int64_t>(r) * p.nc32 + grp] + c_row[r]);
        const float b = expf(m);   // 0 when every row of the block has g = 0
        atomicMax(reinterpret_cast<int*>(p.gmax) + grp, __float_as_int(b));
    }
}

cudaError_t launch_f8_group_max(const ChunkParams& p, int sm_count, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(p.gmax, 0, static_cast<size_t>(p.nc32) * sizeof(float), st);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(p.tokpos, 0xFF, static_cast<size_t>(p.V) * sizeof(int), st);
    if (e != cudaSuccess) return e;
    int blocks = (p.R + kF8GroupRows - 1) / kF8GroupRows;
    if (blocks < 1) blocks = 1;
    (void)sm_count;
    k_f8_group_max<<<blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

// two 8-bit codes of x0 (low byte) and x1 (high byte), saturating
__device__ __forceinline__ uint32_t f8x2(float x0, float x1, bool e5m2) {
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, e5m2 ? __NV_E5M2 : __NV_E4M3));
}

// In place of the 16-bit dlogits pass: from the kept exponentials e = exp(z -
// m_grp) (bf16) write the codes of P = g e exp(m_grp - lse) twice,
//   qa = P * 448 / (|g| exp(zmax - lse)) = sign(g) 448 e exp(m_grp - zmax)   (per row)
//   qb = P * 448 / gmax[grp]                                                 (per group)
// Columns past V and rows past the chunk's last (to the next multiple of 128)
// get code 0.
// 32-byte global load / store (one whole L2 sector per thread); 32-byte aligned addresses
__device__ __forceinline__ void ld_sector(const void* a, uint32_t (&v)[8]) {
    asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "l"(a));
}

__device__ __forceinline__ void st_sector(void* a, const uint32_t (&v)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(a), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__global__ void __launch_bounds__(kTransformThreads) k_transform_f8(const ChunkParams p) {
    if (p.chunk >= p.counts[C_NCHUNKS]) return;
    const int rc = p.counts[C_CHUNK_ROWS];
    const int c0 = p.chunk * rc;
    const int n_c = min(rc, p.counts[C_NVALID] - c0);
    const int n_fill = min(p.R, (n_c + kBM - 1) / kBM * kBM);
    // one 32-column group per thread and step (its two scale factors are the group's):
    // 64 bytes of exponentials in, 32 bytes of each code out, all as whole 32-byte sectors
    // (the buffers are 256-byte aligned and V_pad is a multiple of 64)
    const int ngrp = p.V_pad / 32;
    const bool e5 = p.e5m2 != 0;
    for (int slot = blockIdx.x; slot < n_fill; slot += gridDim.x) {
        const uint16_t* erow = p.dS + static_cast<int64_t>(slot) * p.V_pad;
        uint8_t* arow = p.qa + static_cast<int64_t>(slot) * p.V_pad;
        uint8_t* brow = p.qb + static_cast<int64_t>(slot) * p.V_pad;
        if (slot >= n_c) {
            const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            for (int grp = threadIdx.x; grp < ngrp; grp += kTransformThreads) {
                st_sector(arow + 32 * grp, z);
                st_sector(brow + 32 * grp, z);
            }
            continue;
        }
        const int t = p.rows[c0 + slot];
        if (!GRPO_DCHECK(t >= 0 && t < p.N, p.status)) continue;
        const float g = p.gco[t];
        const float lse = p.lse[t];
        const float zmax = p.rmax[t];
        const float sa = g == 0.f ? 0.f : copysignf(448.f, g);
        const float* mrow = p.mx + static_cast<int64_t>(slot) * p.nc32;
        for (int grp = threadIdx.x; grp < ngrp; grp += kTransformThreads) {
            const int v0 = grp * 32;
            uint32_t oa[8], ob[8];
            if (v0 >= p.V) {
#pragma unroll
                for (int j = 0; j < 8; ++j) oa[j] = ob[j] = 0u;
            } else {
                const float m = mrow[grp];
                const float ca = sa * expf(m - zmax);
                const float gm = p.gmax[grp];
                const float cb = gm > 0.f ? g * expf(m - lse) * (448.f / gm) : 0.f;
                uint32_t u[2][8];
                ld_sector(erow + 32 * grp, u[0]);
                ld_sector(erow + 32 * grp + 16, u[1]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w[4] = {u[j >> 1][4 * (j & 1)], u[j >> 1][4 * (j & 1) + 1],
                                           u[j >> 1][4 * (j & 1) + 2], u[j >> 1][4 * (j & 1) + 3]};
                    uint32_t pa[4], pb[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int v = v0 + 8 * j + 2 * k;
                        const float e0 = v < p.V ? __uint_as_float(w[k] << 16) : 0.f;
                        const float e1 = v + 1 < p.V ? __uint_as_float(w[k] & 0xFFFF0000u) : 0.f;
                        pa[k] = f8x2(ca * e0, ca * e1, e5);
                        pb[k] = f8x2(cb * e0, cb * e1, e5);
                    }
                    oa[2 * j] = pa[0] | (pa[1] << 16);
                    oa[2 * j + 1] = pa[2] | (pa[3] << 16);
                    ob[2 * j] = pb[0] | (pb[1] << 16);
                    ob[2 * j + 1] = pb[2] | (pb[3] << 16);
                }
            }
            st_sector(arow + 32 * grp, oa);
            st_sector(brow + 32 * grp, ob);
        }
    }
}

cudaError_t launch_transform_f8(const ChunkParams& p, int sm_count, cudaStream_t st) {
    int blocks = p.R;
    if (blocks > sm_count * 8) blocks = sm_count * 8;
    k_transform_f8<<<blocks, kTransformThreads, 0, st>>>(p);
    return cudaGetLastError();
}

// Every chunk's (token << 32 | slot) keys in ascending order, one block per
// chunk, by a bitonic sort of the next power of two >= R keys in the block's
// shared memory (padding keys sort last).  Chunk c's keys go to keys[c * R ..].
// The dW epilogue finds the rows of a vocabulary row among them.
__global__ void __launch_bounds__(1024) k_sort_keys(const ChunkParams p, int n_pow2) {
    extern __shared__ unsigned long long keys_sh[];
    const int chunk = blockIdx.x;
    if (chunk >= p.counts[C_NCHUNKS]) return;
    const int rc = p.counts[C_CHUNK_ROWS];
    const int c0 = chunk * rc;
    const int n_c = min(rc, p.counts[C_NVALID] - c0);
    for (int i = threadIdx.x; i < n_pow2; i += blockDim.x) {
        unsigned long long k = ~0ull;
        if (i < n_c) {
            const int t = p.rows[c0 + i];
            const int tok = GRPO_DCHECK(t >= 0 && t < p.N, p.status) ? p.tokens[t] : 0;
            k = (static_cast<unsigned long long>(static_cast<uint32_t>(tok)) << 32) | static_cast<uint32_t>(i);
        }
        keys_sh[i] = k;
    }
    __syncthreads();
    for (int size = 2; size <= n_pow2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < n_pow2; i += blockDim.x) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool up = (i & size) == 0;
                    const unsigned long long a = keys_sh[i], b = keys_sh[j];
                    if ((a > b) == up) {
                        keys_sh[i] = b;
                        keys_sh[j] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    unsigned long long* out = p.keys + static_cast<int64_t>(chunk) * p.R;
    for (int i = threadIdx.x; i < n_c && i < p.R; i += blockDim.x) out[i] = keys_sh[i];
}

cudaError_t launch_sort_keys(const ChunkParams& p, int max_chunks, cudaStream_t st) {
    int n_pow2 = 1;
    while (n_pow2 < p.R) n_pow2 <<= 1;
    if (n_pow2 > kF8SortMax) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(n_pow2) * sizeof(unsigned long long);
    cudaError_t e = cudaFuncSetAttribute(k_sort_keys, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    k_sort_keys<<<max_chunks > 0 ? max_chunks : 1, 1024, smem, st>>>(p, n_pow2);
    return cudaGetLastError();
}

__global__ void k_zero_masked_rows(const uint8_t* __restrict__ mask, int64_t N, int vec_per_row,
                                   uint4* __restrict__ dH) {
    const int64_t total = N * vec_per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / vec_per_row;
        if (!mask[t]) dH[i] = make_uint4(0, 0, 0, 0);
    }
}

cudaError_t launch_zero_masked_rows(const uint8_t* mask, int64_t N, int d, void* dH, int sm_count, cudaStream_t st) {
    const int vpr = d / 8;
    const int64_t total = N * vpr;
    int blocks = static_cast<int>((total + 255) / 256);
    if (blocks > sm_count * 16) blocks = sm_count * 16;
    if (blocks < 1) blocks = 1;
    k_zero_masked_rows<<<blocks, 256, 0, st>>>(mask, N, vpr, static_cast<uint4*>(dH));
    return cudaGetLastError();
}

// found_inf <- 0; dW <- 0 when no row is masked in (no backward chunk runs then)
__global__ void k_clear_grads(const int* __restrict__ counts, int* found_inf, float4* __restrict__ dW, int64_t n4) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *found_inf = 0;
    if (counts[C_NVALID] != 0) return;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        dW[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

cudaError_t launch_clear_grads(const int* counts, int* found_inf, float* dW, int64_t n, int sm_count,
                               cudaStream_t st) {
    const int64_t n4 = n / 4;
    int blocks = static_cast<int>((n4 + 255) / 256);
    if (blocks > sm_count * 8) blocks = sm_count * 8;
    if (blocks < 1) blocks = 1;
    k_clear_grads<<<blocks, 256, 0, st>>>(counts, found_inf, reinterpret_cast<float4*>(dW), n4);
    return cudaGetLastError();
}

}  // namespace grpo
