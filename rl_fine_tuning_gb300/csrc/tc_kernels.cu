// Tensor-core kernels of the linear GRPO loss (tcgen05 + TMEM, fed by TMA).
//
// SM-pair kernels (tcgen05.mma.cta_group::2, M = 256: one 128-row A tile per
// CTA, the 256-wide B tile split between them), one backward chunk per launch:
//   grpo_fwd_pair_kernel  z = H . W^T for the chunk's policy rows (leader CTA)
//         and reference rows (peer CTA) of one 128-row tile, both halves of
//         the MMA reading the same W stage; the epilogue keeps a running
//         (max, sum exp) per row and picks out z[tok] -- the logits are never
//         written anywhere ("Long-context GRPO", section 2: the linear
//         algorithm; section 4: the logsumexp trick).  When a backward
//         follows, the leader also keeps exp(z - running max) in bf16 and the
//         running max per 32 columns, which a streaming pass later turns into
//         the dlogits  s * g_t * (onehot(tok_t) - softmax(z_t)).
//   grpo_fwd_pair_e4m3_kernel, grpo_fwd_pair_e5m2_kernel  the same forward
//         on 8-bit inputs (kind::f8f6f4), scaled by the per-tensor scales.
//   grpo_dh_pair_kernel   dH[rows] = (1/N_valid) * dlogits . W        (K = vocabulary)
//   grpo_dh_pair_wide_kernel  the same in 512-column units: one staged
//         dlogits tile feeds two 256-wide d tiles, the whole tensor memory
//         one accumulator (where those units divide evenly over the pairs)
//   grpo_dw_pair_kernel   dW      += (1/N_valid) * dlogits^T . H_pol  (K = chunk rows; H_pol from
//         the transposed compact rows, so its operand is K-major)
//   grpo_dh_pair_{,wide_}{e4m3,e5m2}_kernel, grpo_dw_pair_{e4m3,e5m2}_kernel
//         the backward on 8-bit codes (kind::f8f6f4, MN-major 8-bit operands):
//         the dlogits' softmax part as codes scaled per row (dH) or per 32
//         vocabulary rows (dW), the one-hot part added exactly in the epilogue
// Single-SM kernel (tcgen05.mma.cta_group::1, M = 128):
//   grpo_fwd_lse_kernel   the forward over row tiles of h_pol / h_ref (the
//         workspace-free entry point), policy and reference MMAs sharing B.
//
// One persistent CTA per SM, 6 warps:
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM allocator + MMA issuer (one lane; in a pair, the leader's)
//   warps 2..5  epilogue; warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31,
//               i.e. one accumulator row per thread.
// Stages: smem ring of kStages K-slices (64 elements = one 128-byte swizzle
// span; 128 for 8-bit operands), full/empty mbarriers; accumulators:
// double-buffered in TMEM (except the single-SM forward, whose two
// accumulators are the policy and reference tiles, and the 512-column dH
// units) with acc_full/acc_empty mbarriers, so the epilogue of one tile
// overlaps the MMAs of the next.
#include <cmath>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace grpo {

constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

// Operand layouts in shared memory (all 128-byte swizzled, as TMA writes them
// with CU_TENSOR_MAP_SWIZZLE_128B):
//   K-major  [rows][64 K-elements]: row r at r*128 B; 8-row groups 1024 B apart
//            (SBO = 1024).  K sub-step kk (16 elements) = +32 B.
//   MN-major [64 K-rows][64 MN-elements] boxes of 8 KB; box j holds MN
//            elements 64j..64j+63 (LBO = 8192); 8-K-row groups 1024 B apart
//            (SBO = 1024).  K sub-step kk = +2048 B.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t a) { return make_sdesc_sw128(a, 16, 1024); }
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t a) { return make_sdesc_sw128(a, 8192, 1024); }

constexpr int kUnitSlots = 4;   // work units published ahead by the producer

struct Smem {
    uint8_t* stages;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* acc_full;
    uint64_t* acc_empty;
    uint64_t* drain;
    uint64_t* unit_full;
    uint64_t* unit_empty;
    uint32_t* tmem_slot;
    volatile int* abort_flag;
    volatile int* unit_id;
    // [0] K-stages whose TMA loads this CTA's producer issued, [1] K-stages the
    // MMA lane consumed, [2] 1 once every issued load is known to have landed
    volatile int* ld_count;
};

template <int kStages, int kStageBytes>
__device__ __forceinline__ Smem carve_smem(uint8_t* raw) {
    Smem s;
    const uint32_t a = smem_u32(raw);
    uint8_t* base = raw + ((1024u - (a & 1023u)) & 1023u);
    s.stages = base;
    s.full = reinterpret_cast<uint64_t*>(base + kStages * kStageBytes);
    s.empty = s.full + kStages;
    s.acc_full = s.empty + kStages;
    s.acc_empty = s.acc_full + 2;
    s.drain = s.acc_empty + 2;
    s.unit_full = s.drain + 1;
    s.unit_empty = s.unit_full + kUnitSlots;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.unit_empty + kUnitSlots);
    s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
    s.unit_id = s.abort_flag + 1;
    s.ld_count = s.unit_id + kUnitSlots;
    return s;
}

template <class T>
constexpr int smem_bytes() {
    return T::kStages * T::kStageBytes + 1024 + 512;
}

// After an abort, wait (at most kInflightNs in all) for the K-stages whose loads
// were issued but not consumed, phases used .. issued-1 of the full barriers,
// to complete.  Returns true when all of them did.
constexpr unsigned long long kInflightNs = 2ull * 1000ull * 1000ull;   // 2 ms

template <int kStages>
__device__ __forceinline__ bool wait_inflight(uint64_t* full, int used, int issued) {
    const uint64_t t0 = globaltimer();
    for (int i = used; i < issued; ++i) {
        const uint32_t a = smem_u32(&full[i % kStages]);
        const uint32_t parity = static_cast<uint32_t>(i / kStages) & 1u;
        while (!mbar_try_wait(a, parity))
            if (globaltimer() - t0 > kInflightNs) return false;
    }
    return true;
}

__device__ __forceinline__ uint16_t f32_to_16(float x, bool bf16) {
    if (bf16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
    return __half_as_ushort(__float2half_rn(x));
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
    return static_cast<uint32_t>(f32_to_16(a, bf16)) | (static_cast<uint32_t>(f32_to_16(b, bf16)) << 16);
}

// non-finite check of a packed pair of fp16 values (exponent all ones)
__device__ __forceinline__ bool half2_nonfinite(uint32_t u) {
    return ((u & 0x7C00u) == 0x7C00u) || ((u & 0x7C000000u) == 0x7C000000u);
}

// ====================================================================== traits
// Each traits class describes one kernel: its schedule of work units, the TMA
// loads of one K-stage, the MMAs of one K-stage and the epilogue.

struct FwdT {
    static constexpr int kStages = 3;
    static constexpr int kStageBytes = 2 * 16384 + 32768;   // A_pol, A_ref (128x64), B (256x64)
    static constexpr int kAccBufs = 1;
    static constexpr int kAccStride = 0;
    using Params = FwdParams;
    struct Sched {
        int n_units, ks, n_tiles;
    };
    struct Coord {
        int t0, n0;
    };
    struct Epi {
        float m[2], s[2], zt[2];
        int tok, t, split;
        bool valid, found;
    };

    // unit = tile * S + split.  Tiles are the forward row tiles over
    // h_pol/h_ref (runs of masked-in rows).
    __device__ static bool setup(const Params& p, Sched& sc) {
        sc.n_tiles = p.counts[C_NTILES];
        sc.n_units = sc.n_tiles * p.S;
        sc.ks = p.d / kBK;
        return sc.n_units > 0;
    }
    __device__ static int tile_of(const Params& p, int unit) { return unit / p.S; }
    __device__ static int items(const Params& p, const Sched&, int unit) {
        const int s = unit % p.S;
        const int nb = s * p.nps;
        const int ne = min(nb + p.nps, p.n_ntiles);
        return max(ne - nb, 0);
    }
    __device__ static int ksteps(const Params&, const Sched& sc, int) { return sc.ks; }
    __device__ static Coord coord(const Params& p, const Sched&, int unit, int item) {
        Coord c;
        c.t0 = p.tiles[tile_of(p, unit)].x;
        c.n0 = ((unit % p.S) * p.nps + item) * kBN;
        return c;
    }
    __device__ static uint32_t tx_bytes(const Params&, const Sched&, const Coord&) { return kStageBytes; }
    __device__ static void load(const Params&, const Sched&, const Coord& c, int k, uint8_t* st, uint64_t* bar,
                                const CUtensorMap* mA, const CUtensorMap* mA2, const CUtensorMap* mB) {
        tma_load_2d(mA, bar, st, k * kBK, c.t0);
        tma_load_2d(mA2, bar, st + 16384, k * kBK, c.t0);
        tma_load_2d(mB, bar, st + 32768, k * kBK, c.n0);
    }
    template <bool kBf16>
    __device__ static void mma(uint32_t st, uint32_t acc, bool first) {
        constexpr uint32_t idesc = make_idesc_f16(128, 256, kBf16, false, false);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t b = desc_kmajor(st + 32768 + kk * 32);
            const uint32_t accum = (first && kk == 0) ? 0u : 1u;
            umma_f16(acc, desc_kmajor(st + kk * 32), b, idesc, accum);
            umma_f16(acc + 256, desc_kmajor(st + 16384 + kk * 32), b, idesc, accum);
        }
    }
    __device__ static void epi_begin(const Params& p, const Sched&, int unit, int row, Epi& e) {
        const int2 tl = p.tiles[tile_of(p, unit)];
        e.t = tl.x + row;
        e.valid = row < tl.y && GRPO_DCHECK(e.t >= 0 && e.t < p.N, p.status);
        if (!e.valid) e.t = 0;
        e.tok = e.valid ? p.tokens[e.t] : -1;
        e.split = unit % p.S;
        e.m[0] = e.m[1] = -INFINITY;
        e.s[0] = e.s[1] = 0.f;
        e.zt[0] = e.zt[1] = 0.f;
        e.found = false;
    }
    template <bool kBf16>
    __device__ static void epi_item(const Params& p, const Sched&, int unit, int item, uint32_t tacc, Epi& e) {
        const int n0 = ((unit % p.S) * p.nps + item) * kBN;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
#pragma unroll 1
            for (int c = 0; c < kBN / 32; ++c) {
                const int col0 = n0 + c * 32;
                if (col0 >= p.V) break;
                float v[32];
                tmem_ld32(tacc + w * 256 + c * 32, v);
                const int nvalid = p.V - col0;
                if (nvalid < 32) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j >= nvalid) v[j] = -INFINITY;
                }
                float cmax = v[0];
#pragma unroll
                for (int j = 1; j < 32; ++j) cmax = fmaxf(cmax, v[j]);
                const float m_new = fmaxf(e.m[w], cmax);
                const float mb = m_new * kLog2e;
                const bool hit = static_cast<unsigned>(e.tok - col0) < 32u;
                if (__any_sync(0xffffffffu, hit)) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (e.tok == col0 + j) e.zt[w] = v[j];
                    if (hit) e.found = true;
                }
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    v[j] = fast_exp2(fmaf(v[j], kLog2e, -mb));
                    acc += v[j];
                }
                e.s[w] = fmaf(e.s[w], fast_exp2(fmaf(e.m[w], kLog2e, -mb)), acc);
                e.m[w] = m_new;
            }
        }
    }
    __device__ static void epi_end(const Params& p, const Sched&, int, Epi& e) {
        if (!e.valid) return;
        p.part[static_cast<int64_t>(e.t) * p.S + e.split] = make_float4(e.m[0], e.s[0], e.m[1], e.s[1]);
        if (e.found) p.zt[e.t] = make_float2(e.zt[0], e.zt[1]);
    }
};

// chunk bookkeeping shared by the backward kernels
struct ChunkSched {
    int n_units, ks, c0, n_c, n_mt, n_nt, n_g, C;
    float winv;
};

__device__ __forceinline__ bool chunk_setup(const ChunkParams& p, ChunkSched& sc, int C) {
    if (p.chunk >= p.counts[C_NCHUNKS]) return false;
    const int rc = p.counts[C_CHUNK_ROWS];
    sc.C = C;
    sc.c0 = p.chunk * rc;
    sc.n_c = min(rc, p.counts[C_NVALID] - sc.c0);
    sc.n_mt = (sc.n_c + kBM - 1) / kBM;
    sc.winv = __int_as_float(p.counts[C_WINV]);
    return sc.n_c > 0;
}

// ====================================================================== engine

template <class T, bool kBf16>
__device__ __forceinline__ void tc_body(const typename T::Params& p, const CUtensorMap& mA, const CUtensorMap& mA2,
                                        const CUtensorMap& mB) {
    extern __shared__ uint8_t smem_raw[];
    typename T::Sched sc;
    if (!T::setup(p, sc)) return;
    if (static_cast<int>(blockIdx.x) >= sc.n_units) return;   // no work for this CTA: leave before touching TMEM
    // CTAs take work units from a per-launch counter
    int* const sched = p.sched;

    Smem sm = carve_smem<T::kStages, T::kStageBytes>(smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int* status = p.status;

    if (threadIdx.x == 0) {
        for (int s = 0; s < T::kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);    // released by the MMA commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.acc_full[b], 1);
            mbar_init(&sm.acc_empty[b], 4);
        }
        for (int u = 0; u < kUnitSlots; ++u) {
            mbar_init(&sm.unit_full[u], 1);
            mbar_init(&sm.unit_empty[u], 5);   // the MMA lane and the four epilogue warps
        }
        mbar_init(sm.drain, 1);
        *sm.abort_flag = 0;
        sm.ld_count[0] = sm.ld_count[1] = sm.ld_count[2] = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&mA);
        tma_prefetch_desc(&mA2);
        tma_prefetch_desc(&mB);
    }
    if (warp == 1) {
        tmem_alloc(sm.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm.tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0, us = 0, n_issued = 0;
            uint32_t ph = 0, uph = 0;
            while (true) {
                const int unit = atomicAdd(sched, 1);
                // publish the unit to the MMA and epilogue roles
                if (!mbar_wait(&sm.unit_empty[us], uph ^ 1u, sm.abort_flag, status)) goto producer_done;
                sm.unit_id[us] = unit;
                mbar_arrive(&sm.unit_full[us]);
                if (++us == kUnitSlots) {
                    us = 0;
                    uph ^= 1u;
                }
                if (unit >= sc.n_units) break;
                const int n_items = T::items(p, sc, unit);
                const int ks = T::ksteps(p, sc, unit);
                for (int item = 0; item < n_items; ++item) {
                    const typename T::Coord c = T::coord(p, sc, unit, item);
                    const uint32_t bytes = T::tx_bytes(p, sc, c);
                    for (int k = 0; k < ks; ++k) {
                        if (!mbar_wait(&sm.empty[s], ph ^ 1u, sm.abort_flag, status)) goto producer_done;
                        uint8_t* st = sm.stages + s * T::kStageBytes;
                        mbar_arrive_expect_tx(&sm.full[s], bytes);
                        T::load(p, sc, c, k, st, &sm.full[s], &mA, &mA2, &mB);
                        ++n_issued;
                        if (++s == T::kStages) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                }
            }
        producer_done:
            sm.ld_count[0] = n_issued;
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0, us = 0, n_used = 0;
            uint32_t ph = 0, uph = 0;
            int it = 0;
            while (true) {
                if (!mbar_wait(&sm.unit_full[us], uph, sm.abort_flag, status)) goto mma_done;
                const int unit = sm.unit_id[us];
                mbar_arrive(&sm.unit_empty[us]);
                if (++us == kUnitSlots) {
                    us = 0;
                    uph ^= 1u;
                }
                if (unit >= sc.n_units) break;
                const int n_items = T::items(p, sc, unit);
                const int ks = T::ksteps(p, sc, unit);
                for (int item = 0; item < n_items; ++item, ++it) {
                    const int b = T::kAccBufs == 1 ? 0 : (it & 1);
                    const uint32_t aph = static_cast<uint32_t>(T::kAccBufs == 1 ? it : (it >> 1)) & 1u;
                    if (!mbar_wait(&sm.acc_empty[b], aph ^ 1u, sm.abort_flag, status)) goto mma_done;
                    tc_fence_after();
                    const uint32_t acc = tmem + b * T::kAccStride;
                    for (int k = 0; k < ks; ++k) {
                        if (!mbar_wait(&sm.full[s], ph, sm.abort_flag, status)) goto mma_done;
                        ++n_used;
                        tc_fence_after();
                        T::template mma<kBf16>(smem_u32(sm.stages + s * T::kStageBytes), acc, k == 0);
                        umma_commit(&sm.empty[s]);
                        if (++s == T::kStages) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    umma_commit(&sm.acc_full[b]);
                }
            }
        mma_done:
            sm.ld_count[1] = n_used;
            // every issued MMA (and every commit it feeds) must have finished
            // before TMEM is released
            umma_commit(sm.drain);
            {
                const uint32_t a = smem_u32(sm.drain);
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(a, 0)) {
                    if (globaltimer() - t0 > kWaitTimeoutNs) {
                        atomicCAS(status, 0, GRPO_ERR_TIMEOUT);
                        break;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        const int row = lane + 32 * (warp & 3);
        const uint32_t tq = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        int it = 0, us = 0;
        uint32_t uph = 0;
        while (true) {
            if (!mbar_wait(&sm.unit_full[us], uph, sm.abort_flag, status)) goto epi_done;
            const int unit = sm.unit_id[us];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.unit_empty[us]);
            if (++us == kUnitSlots) {
                us = 0;
                uph ^= 1u;
            }
            if (unit >= sc.n_units) break;
            const int n_items = T::items(p, sc, unit);
            typename T::Epi e;
            T::epi_begin(p, sc, unit, row, e);
            for (int item = 0; item < n_items; ++item, ++it) {
                const int b = T::kAccBufs == 1 ? 0 : (it & 1);
                const uint32_t aph = static_cast<uint32_t>(T::kAccBufs == 1 ? it : (it >> 1)) & 1u;
                if (!mbar_wait(&sm.acc_full[b], aph, sm.abort_flag, status)) goto epi_done;
                tc_fence_after();
                T::template epi_item<kBf16>(p, sc, unit, item, tq + b * T::kAccStride, e);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.acc_empty[b]);
            }
            T::epi_end(p, sc, unit, e);
        }
    epi_done:;
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    // after an abort, the loads still in flight land on this CTA's own full barriers
    if (*sm.abort_flag) {
        if (threadIdx.x == 0)
            sm.ld_count[2] = wait_inflight<T::kStages>(sm.full, sm.ld_count[1], sm.ld_count[0]) ? 1 : 0;
        __syncthreads();
        if (!sm.ld_count[2]) abort_grace(sm.abort_flag);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ====================================================================== CTA-pair kernels
// The same stages on pairs of SMs with M=256 tcgen05 MMAs (cta_group::2): each
// CTA of a pair holds its own 128-row A tile and half of the 256-column B
// tile, so per SM a K-stage is 32 KB of shared memory instead of 48-64 KB, and
// its tensor memory holds a double-buffered 128x256 accumulator.

// Work-unit orders.  A unit is a pair (a, b); the a-indices are visited in
// groups of G: all b of a group run before the next group starts, and within a
// group the a-indices are fastest.  With G = 1 the b-index is fastest.  The
// group sizes were chosen by timing on GB300 (19 row tiles per group for the
// chunk forward: each W tile is then shared in L2 by 19 tiles).
constexpr int kFwdGroup = 19;   // chunk forward: a = 128-row tile, b = vocabulary split (19 divides 38 and 76)
constexpr int kDhGroup = 1;     // dH: a = pair of 128-row tiles, b = 256-wide d tile
constexpr int kDwGroup = 1;     // dW: a = pair of 128-row vocabulary tiles, b = 256-wide d tile

__device__ __forceinline__ void decode_grouped(int unit, int n_a, int n_b, int G, int* a, int* b) {
    const int full = (n_a / G) * G;
    if (unit < full * n_b) {
        const int gi = unit / (G * n_b);
        const int r = unit - gi * G * n_b;
        *b = r / G;
        *a = gi * G + (r - *b * G);
    } else {
        const int u2 = unit - full * n_b;
        const int g_last = n_a - full;
        *b = u2 / g_last;
        *a = full + (u2 - *b * g_last);
    }
}

__device__ __forceinline__ void decode_tile_split(int unit, int n_mt, int S, int* mt, int* split) {
    decode_grouped(unit, n_mt, S, kFwdGroup, mt, split);
}

// Forward of one chunk: the leader's A rows are the policy tile, the peer's the
// reference tile of the same 128 compact rows; the leader also keeps the
// policy exponentials for the backward.
struct FwdPairT {
    static constexpr int kStages = 7;
    static constexpr int kStageBytes = 16384 + 16384;   // A (128x64), B half (128x64)
    using Params = FwdParams;
    struct Sched {
        int n_units, ks, n_mt, c0, n_c;
    };
    struct Coord {
        int m0, n0;
    };
    struct Epi {
        float m, s, zt;
        int tok, t, split, slot;
        bool valid, found;
    };
    __device__ static bool setup(const Params& p, Sched& sc) {
        if (p.chunk >= p.counts[C_NCHUNKS]) return false;
        const int rc = p.counts[C_CHUNK_ROWS];
        sc.c0 = p.chunk * rc;
        sc.n_c = min(rc, p.counts[C_NVALID] - sc.c0);
        sc.n_mt = (sc.n_c + kBM - 1) / kBM;
        sc.n_units = sc.n_mt * p.S;
        sc.ks = p.d / kBK;
        return sc.n_units > 0;
    }
    __device__ static int items(const Params& p, const Sched& sc, int unit) {
        int mt, split;
        decode_tile_split(unit, sc.n_mt, p.S, &mt, &split);
        const int nb = split * p.nps;
        return max(min(nb + p.nps, p.n_ntiles) - nb, 0);
    }
    __device__ static int ksteps(const Params&, const Sched& sc, int) { return sc.ks; }
    __device__ static Coord coord(const Params& p, const Sched& sc, int unit, int item, int) {
        int mt, split;
        decode_tile_split(unit, sc.n_mt, p.S, &mt, &split);
        return Coord{mt * kBM, (split * p.nps + item) * kBN};
    }
    __device__ static uint32_t tx_bytes(const Params&, const Sched&, const Coord&) { return 2 * kStageBytes; }
    __device__ static void load(const Params&, const Sched&, const Coord& c, int k, uint8_t* st, uint32_t bar,
                                const CUtensorMap* mA, const CUtensorMap* mA2, const CUtensorMap* mB, int rank) {
        tma_load_2d_pair(rank == 0 ? mA : mA2, bar, st, k * kBK, c.m0);
        tma_load_2d_pair(mB, bar, st + 16384, k * kBK, c.n0 + rank * 128);
    }
    template <bool kBf16>
    __device__ static void mma(uint32_t st, uint32_t acc, bool first) {
        constexpr uint32_t idesc = make_idesc_f16(256, 256, kBf16, false, false);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            umma_pair_f16(acc, desc_kmajor(st + kk * 32), desc_kmajor(st + 16384 + kk * 32), idesc,
                          (first && kk == 0) ? 0u : 1u);
    }
    __device__ static void epi_begin(const Params& p, const Sched& sc, int unit, int, int row, Epi& e) {
        int mt, split;
        decode_tile_split(unit, sc.n_mt, p.S, &mt, &split);
        e.slot = mt * kBM + row;
        e.valid = e.slot < sc.n_c && GRPO_DCHECK(e.slot < p.R, p.status);
        e.t = e.valid ? p.rows[sc.c0 + e.slot] : 0;
        if (e.valid && !GRPO_DCHECK(e.t >= 0 && e.t < p.N, p.status)) e.valid = false;
        e.tok = e.valid ? p.tokens[e.t] : -1;
        e.split = split;
        e.m = -INFINITY;
        e.s = 0.f;
        e.zt = 0.f;
        e.found = false;
    }
    template <bool kBf16>
    __device__ static void epi_item(const Params& p, const Sched&, int unit, int item, int rank, uint32_t tacc,
                                    Epi& e) {
        const int n0 = (e.split * p.nps + item) * kBN;
        (void)unit;
        const bool keep = rank == 0 && p.E != nullptr && e.valid;
        uint16_t* erow = keep ? p.E + static_cast<int64_t>(e.slot) * p.V_pad : nullptr;
        float* mrow = keep ? p.mx + static_cast<int64_t>(e.slot) * p.nc32 : nullptr;
        // running maxima of the tile's eight 32-column groups, stored together at the end
        float mv[kBN / 32];
#pragma unroll
        for (int j = 0; j < kBN / 32; ++j) mv[j] = 0.f;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
            const int col0 = n0 + c * 32;
            if (col0 >= p.V) break;
            float v[32];
            tmem_ld32(tacc + c * 32, v);
            const float zs = p.zscale[rank];
            if (zs != 1.f) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= zs;
            }
            const int nvalid = p.V - col0;
            if (nvalid < 32) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j >= nvalid) v[j] = -INFINITY;
            }
            float cmax = v[0];
#pragma unroll
            for (int j = 1; j < 32; ++j) cmax = fmaxf(cmax, v[j]);
            const float m_new = fmaxf(e.m, cmax);
            const float mb = m_new * kLog2e;
            const bool hit = static_cast<unsigned>(e.tok - col0) < 32u;
            if (__any_sync(0xffffffffu, hit)) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (e.tok == col0 + j) e.zt = v[j];
                if (hit) e.found = true;
            }
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                v[j] = fast_exp2(fmaf(v[j], kLog2e, -mb));
                acc += v[j];
            }
            e.s = fmaf(e.s, fast_exp2(fmaf(e.m, kLog2e, -mb)), acc);
            e.m = m_new;
            if (keep && GRPO_DCHECK(col0 + 32 <= p.V_pad, p.status)) {
                // 64 bytes of one row as two whole 32-byte sectors
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    st_global_v8(erow + col0 + 16 * h, pack2(v[16 * h], v[16 * h + 1], true),
                                 pack2(v[16 * h + 2], v[16 * h + 3], true), pack2(v[16 * h + 4], v[16 * h + 5], true),
                                 pack2(v[16 * h + 6], v[16 * h + 7], true), pack2(v[16 * h + 8], v[16 * h + 9], true),
                                 pack2(v[16 * h + 10], v[16 * h + 11], true),
                                 pack2(v[16 * h + 12], v[16 * h + 13], true),
                                 pack2(v[16 * h + 14], v[16 * h + 15], true));
#pragma unroll
                for (int j = 0; j < kBN / 32; ++j)
                    if (c == j) mv[j] = m_new;
            }
        }
        // the row pitch of mx is a multiple of 8 groups and n0 of 256 columns: 32-byte aligned
        if (keep && GRPO_DCHECK((n0 >> 5) + kBN / 32 <= p.nc32, p.status))
            st_global_v8(mrow + (n0 >> 5), __float_as_uint(mv[0]), __float_as_uint(mv[1]), __float_as_uint(mv[2]),
                         __float_as_uint(mv[3]), __float_as_uint(mv[4]), __float_as_uint(mv[5]),
                         __float_as_uint(mv[6]), __float_as_uint(mv[7]));
    }
    // the leader writes the policy half of the partials, the peer the reference half
    __device__ static void epi_end(const Params& p, const Sched&, int rank, Epi& e) {
        if (!e.valid || !GRPO_DCHECK(e.split >= 0 && e.split < p.S, p.status)) return;
        float* part = reinterpret_cast<float*>(p.part + static_cast<int64_t>(e.slot) * p.S + e.split);
        *reinterpret_cast<float2*>(part + 2 * rank) = make_float2(e.m, e.s);
        if (e.found) reinterpret_cast<float*>(p.zt + e.t)[rank] = e.zt;
    }
};

// The chunk forward on 8-bit inputs (OCP E4M3, or E5M2 when kE5M2): the same
// tiles, byte for byte (a 128-byte row holds 128 elements), a K-stage of 128
// elements, four K=32 MMAs of kind f8f6f4 per stage, and the per-tensor scales
// applied to the accumulator.
template <bool kE5M2>
struct FwdPairF8T : FwdPairT {
    static constexpr int kStageElems = 128;
    __device__ static bool setup(const Params& p, Sched& sc) {
        if (!FwdPairT::setup(p, sc)) return false;
        sc.ks = p.d / kStageElems;
        return true;
    }
    __device__ static void load(const Params&, const Sched&, const Coord& c, int k, uint8_t* st, uint32_t bar,
                                const CUtensorMap* mA, const CUtensorMap* mA2, const CUtensorMap* mB, int rank) {
        tma_load_2d_pair(rank == 0 ? mA : mA2, bar, st, k * kStageElems, c.m0);
        tma_load_2d_pair(mB, bar, st + 16384, k * kStageElems, c.n0 + rank * 128);
    }
    template <bool>
    __device__ static void mma(uint32_t st, uint32_t acc, bool first) {
        constexpr uint32_t idesc = make_idesc_f8(256, 256, kE5M2);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            umma_pair_f8(acc, desc_kmajor(st + kk * 32), desc_kmajor(st + 16384 + kk * 32), idesc,
                         (first && kk == 0) ? 0u : 1u);
    }
};

struct DhPairT {
    static constexpr int kStages = 7;
    static constexpr int kStageBytes = 16384 + 16384;   // A (128 slots x 64 vocab), B half (64 vocab x 128 d)
    using Params = ChunkParams;
    using Sched = ChunkSched;
    struct Coord {
        int m0, n0;
    };
    struct Epi {
        int unused;
    };
    // unit -> (pair of 128-row tiles, d tile); the CTA of rank r takes m-tile 2*pair + r
    __device__ static bool setup(const Params& p, Sched& sc) {
        if (!chunk_setup(p, sc, 2)) return false;
        sc.n_nt = (p.d + kBN - 1) / kBN;
        sc.n_g = (sc.n_mt + 1) / 2;
        sc.ks = (p.V + kBK - 1) / kBK;
        sc.n_units = sc.n_g * sc.n_nt;
        return true;
    }
    __device__ static void decode(const Sched& sc, int unit, int* pair, int* dt) {
        decode_grouped(unit, sc.n_g, sc.n_nt, kDhGroup, pair, dt);
    }
    __device__ static int mtile(const Sched& sc, int unit, int rank) {
        int pair, dt;
        decode(sc, unit, &pair, &dt);
        return pair * 2 + rank;
    }
    __device__ static int dtile(const Sched& sc, int unit) {
        int pair, dt;
        decode(sc, unit, &pair, &dt);
        return dt;
    }
    __device__ static int items(const Params&, const Sched&, int) { return 1; }
    __device__ static int ksteps(const Params&, const Sched& sc, int) { return sc.ks; }
    __device__ static Coord coord(const Params&, const Sched& sc, int unit, int, int rank) {
        return Coord{mtile(sc, unit, rank) * kBM, dtile(sc, unit) * kBN};
    }
    __device__ static uint32_t tx_bytes(const Params& p, const Sched&, const Coord& c) {
        return 2 * 16384 + 8192 * min(4, (p.d - c.n0) / 64);
    }
    __device__ static void load(const Params& p, const Sched&, const Coord& c, int k, uint8_t* st, uint32_t bar,
                                const CUtensorMap* mA, const CUtensorMap*, const CUtensorMap* mB, int rank) {
        tma_load_2d_pair(mA, bar, st, k * kBK, c.m0);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int col = c.n0 + rank * 128 + 64 * j;
            if (col < p.d) tma_load_2d_pair(mB, bar, st + 16384 + 8192 * j, col, k * kBK);
        }
    }
    template <bool kBf16>
    __device__ static void mma(uint32_t st, uint32_t acc, bool first) {
        constexpr uint32_t idesc = make_idesc_f16(256, 256, kBf16, false, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            umma_pair_f16(acc, desc_kmajor(st + kk * 32), desc_mnmajor(st + 16384 + kk * 2048), idesc,
                          (first && kk == 0) ? 0u : 1u);
    }
    __device__ static void epi_begin(const Params&, const Sched&, int, int, int, Epi&) {}
    template <bool kBf16>
    __device__ static void epi_item(const Params& p, const Sched& sc, int unit, int, int rank, uint32_t tacc, Epi&) {
        const int row = (threadIdx.x & 31) + 32 * ((threadIdx.x >> 5) & 3);
        const int slot = mtile(sc, unit, rank) * kBM + row;
        const int n0 = dtile(sc, unit) * kBN;
        bool valid = slot < sc.n_c;
        if (!__any_sync(0xffffffffu, valid)) return;
        const int t = valid ? p.rows[sc.c0 + slot] : 0;
        if (valid && !GRPO_DCHECK(t >= 0 && t < p.N, p.status)) valid = false;
        uint16_t* out = p.dH + static_cast<int64_t>(t) * p.d;
        bool bad = false;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
            const int col0 = n0 + c * 32;
            if (col0 >= p.d) break;
            float v[32];
            tmem_ld32(tacc + c * 32, v);
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) pk[j / 2] = pack2(v[j] * sc.winv, v[j + 1] * sc.winv, kBf16);
            if (!kBf16) {
#pragma unroll
                for (int j = 0; j < 16; ++j) bad |= half2_nonfinite(pk[j]);
            }
            if (valid) {
                // 64 bytes of one dH row as two whole sectors (dH is 32-byte aligned, d a multiple of 64)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    st_global_v8(out + col0 + 16 * h, pk[8 * h], pk[8 * h + 1], pk[8 * h + 2], pk[8 * h + 3],
                                 pk[8 * h + 4], pk[8 * h + 5], pk[8 * h + 6], pk[8 * h + 7]);
            }
        }
        if (bad && valid) atomicOr(p.found_inf, 1);
    }
    __device__ static void epi_end(const Params&, const Sched&, int, Epi&) {}
};

// dH with 512-column units: one staged 128-row dlogits tile feeds two 256-wide
// d tiles (two M=256 MMAs per K sub-step into the two halves of tensor
// memory), so the dlogits are read half as often and W in half as many waves.
// Used where its units still divide evenly over the SM pairs.
struct DhPairWideT {
    static constexpr int kStages = 4;
    static constexpr int kStageBytes = 16384 + 2 * 16384;   // A (128 slots x 64 vocab), 2 x B half (64 vocab x 128 d)
    static constexpr bool kWideAcc = true;
    using Params = ChunkParams;
    using Sched = ChunkSched;
    struct Coord {
        int m0, n0;
    };
    struct Epi {
        int unused;
    };
    // unit -> (pair of 128-row tiles, 512-wide d tile); the CTA of rank r takes m-tile 2*pair + r
    __device__ static bool setup(const Params& p, Sched& sc) {
        if (!chunk_setup(p, sc, 2)) return false;
        sc.n_nt = (p.d + 2 * kBN - 1) / (2 * kBN);
        sc.n_g = (sc.n_mt + 1) / 2;
        sc.ks = (p.V + kBK - 1) / kBK;
        sc.n_units = sc.n_g * sc.n_nt;
        return true;
    }
    __device__ static int mtile(const Sched& sc, int unit, int rank) { return (unit / sc.n_nt) * 2 + rank; }
    __device__ static int dtile(const Sched& sc, int unit) { return unit % sc.n_nt; }
    __device__ static int items(const Params&, const Sched&, int) { return 1; }
    __device__ static int ksteps(const Params&, const Sched& sc, int) { return sc.ks; }
    __device__ static Coord coord(const Params&, const Sched& sc, int unit, int, int rank) {
        return Coord{mtile(sc, unit, rank) * kBM, dtile(sc, unit) * 2 * kBN};
    }
    __device__ static uint32_t tx_bytes(const Params& p, const Sched&, const Coord& c) {
        uint32_t b = 2 * 16384;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    if (c.n0 + h * kBN + r * 128 + 64 * j < p.d) b += 8192;
        return b;
    }
    __device__ static void load(const Params& p, const Sched&, const Coord& c, int k, uint8_t* st, uint32_t bar,
                                const CUtensorMap* mA, const CUtensorMap*, const CUtensorMap* mB, int rank) {
        tma_load_2d_pair(mA, bar, st, k * kBK, c.m0);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int col = c.n0 + h * kBN + rank * 128 + 64 * j;
                if (col < p.d) tma_load_2d_pair(mB, bar, st + 16384 + 16384 * h + 8192 * j, col, k * kBK);
            }
    }
    template <bool kBf16>
    __device__ static void mma(uint32_t st, uint32_t acc, bool first) {
        constexpr uint32_t idesc = make_idesc_f16(256, 256, kBf16, false, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = desc_kmajor(st + kk * 32);
            const uint32_t accum = (first && kk == 0) ? 0u : 1u;
            umma_pair_f16(acc, a, desc_mnmajor(st + 16384 + kk * 2048), idesc, accum);
            umma_pair_f16(acc + 256, a, desc_mnmajor(st + 32768 + kk * 2048), idesc, accum);
        }
    }
    __device__ static void epi_begin(const Params&, const Sched&, int, int, int, Epi&) {}
    template <bool kBf16>
    __device__ static void epi_item(const Params& p, const Sched& sc, int unit, int, int rank, uint32_t tacc, Epi&) {
        const int row = (threadIdx.x & 31) + 32 * ((threadIdx.x >> 5) & 3);
        const int slot = mtile(sc, unit, rank) * kBM + row;
        const int n0 = dtile(sc, unit) * 2 * kBN;
        bool valid = slot < sc.n_c;
        if (!__any_sync(0xffffffffu, valid)) return;
        const int t = valid ? p.rows[sc.c0 + slot] : 0;
        if (valid && !GRPO_DCHECK(t >= 0 && t < p.N, p.status)) valid = false;
        uint16_t* out = p.dH + static_cast<int64_t>(t) * p.d;
        bool bad = false;
#pragma unroll 1
        for (int c = 0; c < 2 * kBN / 32; ++c) {
            const int col0 = n0 + c * 32;
            if (col0 >= p.d) break;
            float v[32];
            tmem_ld32(tacc + c * 32, v);
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) pk[j / 2] = pack2(v[j] * sc.winv, v[j + 1] * sc.winv, kBf16);
            if (!kBf16) {
#pragma unroll
                for (int j = 0; j < 16; ++j) bad |= half2_nonfinite(pk[j]);
            }
            if (valid) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    st_global_v8(out + col0 + 16 * h, pk[8 * h], pk[8 * h + 1], pk[8 * h + 2], pk[8 * h + 3],
                                 pk[8 * h + 4], pk[8 * h + 5], pk[8 * h + 6], pk[8 * h + 7]);
            }
        }
        if (bad && valid) atomicOr(p.found_inf, 1);
    }
    __device__ static void epi_end(const Params&, const Sched&, int, Epi&) {}
};

struct DwPairT {
    static constexpr int kStages = 7;
    static constexpr int kStageBytes = 16384 + 16384;   // A (64 slots x 128 vocab), B half (128 d x 64 slots)
    using Params = ChunkParams;
    using Sched = ChunkSched;
    struct Coord {
        int v0, n0;
    };
    struct Epi {
        int unused;
    };
    // unit -> (pair of vocabulary tiles, d tile); the CTA of rank r takes vocabulary tile 2*pair + r
    __device__ static bool setup(const Params& p, Sched& sc) {
        if (!chunk_setup(p, sc, 2)) return false;
        sc.n_nt = (p.d + kBN - 1) / kBN;
        sc.n_g = ((p.V + kBM - 1) / kBM + 1) / 2;
        sc.ks = (sc.n_c + kBK - 1) / kBK;
        sc.n_units = sc.n_g * sc.n_nt;
        return true;
    }
    __device__ static void decode(const Sched& sc, int unit, int* pair, int* dt) {
        decode_grouped(unit, sc.n_g, sc.n_nt, kDwGroup, pair, dt);
    }
    __device__ static int vtile(const Sched& sc, int unit, int rank) {
        int pair, dt;
        decode(sc, unit, &pair, &dt);
        return pair * 2 + rank;
    }
    __device__ static int dtile(const Sched& sc, int unit) {
        int pair, dt;
        decode(sc, unit, &pair, &dt);
        return dt;
    }
    __device__ static int items(const Params&, const Sched&, int) { return 1; }
    __device__ static int ksteps(const Params&, const Sched& sc, int) { return sc.ks; }
    __device__ static Coord coord(const Params&, const Sched& sc, int unit, int, int rank) {
        return Coord{vtile(sc, unit, rank) * kBM, dtile(sc, unit) * kBN};
    }
    __device__ static uint32_t tx_bytes(const Params& p, const Sched&, const Coord& c) {
        return 2 * 16384 + 16384 * min(2, (p.d - c.n0 + 127) / 128);
    }
    __device__ static void load(const Params& p, const Sched&, const Coord& c, int k, uint8_t* st, uint32_t bar,
                                const CUtensorMap* mA, const CUtensorMap*, const CUtensorMap* mB, int rank) {
        tma_load_2d_pair(mA, bar, st, c.v0, k * kBK);
        tma_load_2d_pair(mA, bar, st + 8192, c.v0 + 64, k * kBK);
        // B: 128 rows of the transposed compact h_pol (d) x 64 chunk slots (K), K-major
        const int col = c.n0 + rank * 128;
        if (col < p.d) tma_load_2d_pair(mB, bar, st + 16384, k * kBK, col);
    }
    template <bool kBf16>
    __device__ static void mma(uint32_t st, uint32_t acc, bool first) {
        constexpr uint32_t idesc = make_idesc_f16(256, 256, kBf16, true, false);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            umma_pair_f16(acc, desc_mnmajor(st + kk * 2048), desc_kmajor(st + 16384 + kk * 32), idesc,
                          (first && kk == 0) ? 0u : 1u);
    }
    __device__ static void epi_begin(const Params&, const Sched&, int, int, int, Epi&) {}
    template <bool kBf16>
    __device__ static void epi_item(const Params& p, const Sched& sc, int unit, int, int rank, uint32_t tacc, Epi&) {
        const int row = (threadIdx.x & 31) + 32 * ((threadIdx.x >> 5) & 3);
        const int v = vtile(sc, unit, rank) * kBM + row;
        const int n0 = dtile(sc, unit) * kBN;
        const bool valid = v < p.V;
        if (!__any_sync(0xffffffffu, valid)) return;
        const bool first_chunk = p.chunk == 0;
        float* out = p.dW + static_cast<int64_t>(valid ? v : 0) * p.d;
        bool bad = false;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
            const int col0 = n0 + c * 32;
            if (col0 >= p.d) break;
            float x[32];
            tmem_ld32(tacc + c * 32, x);
            if (valid) {
                // 128 bytes of one dW row as four whole sectors (dW is 32-byte aligned)
                float* o = out + col0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float r[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) r[i] = x[8 * j + i] * sc.winv;
                    if (!first_chunk) {
                        float prev[8];
                        ld_global_v8(o + 8 * j, prev);
#pragma unroll
                        for (int i = 0; i < 8; ++i) r[i] += prev[i];
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) bad |= !isfinite(r[i]);
                    st_global_v8(o + 8 * j, __float_as_uint(r[0]), __float_as_uint(r[1]), __float_as_uint(r[2]),
                                 __float_as_uint(r[3]), __float_as_uint(r[4]), __float_as_uint(r[5]),
                                 __float_as_uint(r[6]), __float_as_uint(r[7]));
                }
            }
        }
        if (bad) atomicOr(p.found_inf, 1);
    }
    __device__ static void epi_end(const Params&, const Sched&, int, Epi&) {}
};

// ---------------------------------------------------------------------- 8-bit backward
// The two backward GEMMs on 8-bit codes (kind::f8f6f4, M = 256 pairs, K = 32
// per instruction, a K-stage of 128).  A operand: the codes of P = g softmax
// (the dlogits without their one-hot part); B: the 8-bit W (dH) or the
// chunk's 8-bit h_pol rows (dW).  Each code buffer carries one scale per
// M-row (per dlogit row for dH, per 32-vocabulary-row group for dW), which
// factors out of the K sum; the epilogue applies it and adds the one-hot part
// exactly, from the decoded 8-bit inputs:
//   dH_t = w scale_w (g_t Wc[tok_t] - s_t acc),           s_t = |g_t| exp(zmax_t - lse_t) / 448
//   dW_v = w scale_h (sum_{t: tok_t = v} g_t hc_t - gmax_grp(v) / 448 acc)

// MN-major 8-bit operand: [128 K-rows][128 MN-bytes] boxes of 16 KB; 8-K-row
// groups 1024 B apart (SBO); K sub-step of 32 = +4096 B.
__device__ __forceinline__ uint64_t desc_mnmajor_f8(uint32_t a) { return make_sdesc_sw128(a, 16384, 1024); }

// 32 8-bit codes -> floats (exact)
__device__ __forceinline__ void decode32_f8(const uint8_t* src, bool e5m2, float (&out)[32]) {
    const uint4* q = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint4 u = q[h];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const __nv_fp8x2_storage_t pr = static_cast<__nv_fp8x2_storage_t>((w[j] >> (16 * k)) & 0xFFFFu);
                const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pr, e5m2 ? __NV_E5M2 : __NV_E4M3);
                const float2 f = __half22float2(__half2(hr));
                out[16 * h + 4 * j + 2 * k] = f.x;
                out[16 * h + 4 * j + 2 * k + 1] = f.y;
            }
        }
    }
}

struct DhPairF8T : DhPairT {
    static constexpr int kStageElems = 128;
    __device__ static bool setup(const Params& p, Sched& sc) {
        if (!DhPairT::setup(p, sc)) return false;
        sc.ks = (p.V + kStageElems - 1) / kStageElems;
        return true;
    }
    __device__ static uint32_t tx_bytes(const Params& p, const Sched&, const Coord& c) {
        return 2 * 16384 + 16384 * min(2, (p.d - c.n0) / 128);
    }
    __device__ static void load(const Params& p, const Sched&, const Coord& c, int k, uint8_t* st, uint32_t bar,
                                const CUtensorMap* mA, const CUtensorMap*, const CUtensorMap* mB, int rank) {
        tma_load_2d_pair(mA, bar, st, k * kStageElems, c.m0);
        const int col = c.n0 + rank * 128;
        if (col < p.d) tma_load_2d_pair(mB, bar, st + 16384, col, k * kStageElems);
    }
    template <bool>
    __device__ static void mma(uint32_t st, uint32_t acc, bool first) {
        // the format is a launch parameter: E4M3 here, E5M2 in DhPairF8T5
        mma_fmt<false>(st, acc, first);
    }
    template <bool kE5M2>
    __device__ static void mma_fmt(uint32_t st, uint32_t acc, bool first) {
        constexpr uint32_t idesc = make_idesc_f8(256, 256, kE5M2, false, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            umma_pair_f8(acc, desc_kmajor(st + kk * 32), desc_mnmajor_f8(st + 16384 + kk * 4096), idesc,
                         (first && kk == 0) ? 0u : 1u);
    }
    template <bool>
    __device__ static void epi_item(const Params& p, const Sched& sc, int unit, int, int rank, uint32_t tacc, Epi&) {
        const int row = (threadIdx.x & 31) + 32 * ((threadIdx.x >> 5) & 3);
        const int slot = mtile(sc, unit, rank) * kBM + row;
        const int n0 = dtile(sc, unit) * kBN;
        bool valid = slot < sc.n_c;
        if (!__any_sync(0xffffffffu, valid)) return;
        const int t = valid ? p.rows[sc.c0 + slot] : 0;
        if (valid && !GRPO_DCHECK(t >= 0 && t < p.N, p.status)) valid = false;
        // a token id outside [0, V) has g = 0 (the merge reported it): no W row is read for it
        int tok = valid ? p.tokens[t] : 0;
        const bool tok_ok = tok >= 0 && tok < p.V;
        if (!tok_ok) tok = 0;
        const float g = valid && tok_ok ? p.gco[t] : 0.f;
        const float s_t = valid ? fabsf(g) * expf(p.rmax[t] - p.lse[t]) * (1.f / 448.f) : 0.f;
        const float f = sc.winv * p.scale_w;
        uint16_t* out = p.dH + static_cast<int64_t>(t) * p.d;
        const uint8_t* wrow = p.wq + static_cast<int64_t>(tok) * p.d;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
            const int col0 = n0 + c * 32;
            if (col0 >= p.d) break;
            float v[32];
            tmem_ld32(tacc + c * 32, v);
            if (!valid) continue;
            float wt[32];
            decode32_f8(wrow + col0, p.e5m2 != 0, wt);
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2)
                pk[j / 2] = pack2(f * (g * wt[j] - s_t * v[j]), f * (g * wt[j + 1] - s_t * v[j + 1]), true);
#pragma unroll
            for (int h = 0; h < 2; ++h)
                st_global_v8(out + col0 + 16 * h, pk[8 * h], pk[8 * h + 1], pk[8 * h + 2], pk[8 * h + 3],
                             pk[8 * h + 4], pk[8 * h + 5], pk[8 * h + 6], pk[8 * h + 7]);
        }
    }
};

struct DhPairF8T5 : DhPairF8T {
    template <bool>
    __device__ static void mma(uint32_t st, uint32_t acc, bool first) {
        mma_fmt<true>(st, acc, first);
    }
};

// The 8-bit dH in 512-column units (see DhPairWideT): a K-stage of 128 vocabulary
// rows, two MMAs per K sub-step from one staged code tile, the epilogue of
// DhPairF8T over both 256-column halves.
struct DhPairF8WideT : DhPairWideT {
    static constexpr int kStageElems = 128;
    __device__ static bool setup(const Params& p, Sched& sc) {
        if (!DhPairWideT::setup(p, sc)) return false;
        sc.ks = (p.V + kStageElems - 1) / kStageElems;
        return true;
    }
    __device__ static uint32_t tx_bytes(const Params& p, const Sched&, const Coord& c) {
        uint32_t b = 2 * 16384;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int r = 0; r < 2; ++r)
                if (c.n0 + h * kBN + r * 128 < p.d) b += 16384;
        return b;
    }
    __device__ static void load(const Params& p, const Sched&, const Coord& c, int k, uint8_t* st, uint32_t bar,
                                const CUtensorMap* mA, const CUtensorMap*, const CUtensorMap* mB, int rank) {
        tma_load_2d_pair(mA, bar, st, k * kStageElems, c.m0);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = c.n0 + h * kBN + rank * 128;
            if (col < p.d) tma_load_2d_pair(mB, bar, st + 16384 + 16384 * h, col, k * kStageElems);
        }
    }
    template <bool kE5M2>
    __device__ static void mma_fmt(uint32_t st, uint32_t acc, bool first) {
        constexpr uint32_t idesc = make_idesc_f8(256, 256, kE5M2, false, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = desc_kmajor(st + kk * 32);
            const uint32_t accum = (first && kk == 0) ? 0u : 1u;
            umma_pair_f8(acc, a, desc_mnmajor_f8(st + 16384 + kk * 4096), idesc, accum);
            umma_pair_f8(acc + 256, a, desc_mnmajor_f8(st + 32768 + kk * 4096), idesc, accum);
        }
    }
    template <bool>
    __device__ static void mma(uint32_t st, uint32_t acc, bool first) {
        mma_fmt<false>(st, acc, first);
    }
    template <bool>
    __device__ static void epi_item(const Params& p, const Sched& sc, int unit, int, int rank, uint32_t tacc, Epi&) {
        const int row = (threadIdx.x & 31) + 32 * ((threadIdx.x >> 5) & 3);
        const int slot = mtile(sc, unit, rank) * kBM + row;
        const int n0 = dtile(sc, unit) * 2 * kBN;
        bool valid = slot < sc.n_c;
        if (!__any_sync(0xffffffffu, valid)) return;
        const int t = valid ? p.rows[sc.c0 + slot] : 0;
        if (valid && !GRPO_DCHECK(t >= 0 && t < p.N, p.status)) valid = false;
        // a token id outside [0, V) has g = 0 (the merge reported it): no W row is read for it
        int tok = valid ? p.tokens[t] : 0;
        const bool tok_ok = tok >= 0 && tok < p.V;
        if (!tok_ok) tok = 0;
        const float g = valid && tok_ok ? p.gco[t] : 0.f;
        const float s_t = valid ? fabsf(g) * expf(p.rmax[t] - p.lse[t]) * (1.f / 448.f) : 0.f;
        const float f = sc.winv * p.scale_w;
        uint16_t* out = p.dH + static_cast<int64_t>(t) * p.d;
        const uint8_t* wrow = p.wq + static_cast<int64_t>(tok) * p.d;
#pragma unroll 1
        for (int c = 0; c < 2 * kBN / 32; ++c) {
            const int col0 = n0 + c * 32;
            if (col0 >= p.d) break;
            float v[32];
            tmem_ld32(tacc + c * 32, v);
            if (!valid) continue;
            float wt[32];
            decode32_f8(wrow + col0, p.e5m2 != 0, wt);
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2)
                pk[j / 2] = pack2(f * (g * wt[j] - s_t * v[j]), f * (g * wt[j + 1] - s_t * v[j + 1]), true);
#pragma unroll
            for (int h = 0; h < 2; ++h)
                st_global_v8(out + col0 + 16 * h, pk[8 * h], pk[8 * h + 1], pk[8 * h + 2], pk[8 * h + 3],
                             pk[8 * h + 4], pk[8 * h + 5], pk[8 * h + 6], pk[8 * h + 7]);
        }
    }
};

struct DhPairF8WideT5 : DhPairF8WideT {
    template <bool>
    __device__ static void mma(uint32_t st, uint32_t acc, bool first) {
        mma_fmt<true>(st, acc, first);
    }
};

struct DwPairF8T : DwPairT {
    static constexpr int kStageElems = 128;
    __device__ static bool setup(const Params& p, Sched& sc) {
        if (!DwPairT::setup(p, sc)) return false;
        sc.ks = (sc.n_c + kStageElems - 1) / kStageElems;
        return true;
    }
    __device__ static uint32_t tx_bytes(const Params& p, const Sched&, const Coord& c) {
        return 2 * 16384 + 16384 * min(2, (p.d - c.n0) / 128);
    }
    __device__ static void load(const Params& p, const Sched&, const Coord& c, int k, uint8_t* st, uint32_t bar,
                                const CUtensorMap* mA, const CUtensorMap*, const CUtensorMap* mB, int rank) {
        tma_load_2d_pair(mA, bar, st, c.v0, k * kStageElems);
        const int col = c.n0 + rank * 128;
        if (col < p.d) tma_load_2d_pair(mB, bar, st + 16384, col, k * kStageElems);
    }
    template <bool>
    __device__ static void mma(uint32_t st, uint32_t acc, bool first) {
        mma_fmt<false>(st, acc, first);
    }
    template <bool kE5M2>
    __device__ static void mma_fmt(uint32_t st, uint32_t acc, bool first) {
        constexpr uint32_t idesc = make_idesc_f8(256, 256, kE5M2, true, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            umma_pair_f8(acc, desc_mnmajor_f8(st + kk * 4096), desc_mnmajor_f8(st + 16384 + kk * 4096), idesc,
                         (first && kk == 0) ? 0u : 1u);
    }
    template <bool>
    __device__ static void epi_item(const Params& p, const Sched& sc, int unit, int, int rank, uint32_t tacc, Epi&) {
        const int row = (threadIdx.x & 31) + 32 * ((threadIdx.x >> 5) & 3);
        const int v = vtile(sc, unit, rank) * kBM + row;
        const int n0 = dtile(sc, unit) * kBN;
        const bool valid = v < p.V;
        if (!__any_sync(0xffffffffu, valid)) return;
        const bool first_chunk = p.chunk == 0;
        // the chunk's rows whose sampled token is v: a run of the sorted keys from tokpos[v]
        const int lo = valid ? p.tokpos[v] : -1;
        int n_hit = 0;
        while (lo >= 0 && lo + n_hit < sc.n_c && (p.keys[lo + n_hit] >> 32) == static_cast<unsigned long long>(v))
            ++n_hit;
        const float fb = valid ? p.gmax[v >> 5] * (1.f / 448.f) : 0.f;
        const float f = sc.winv * p.scale_h;
        float* out = p.dW + static_cast<int64_t>(valid ? v : 0) * p.d;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
            const int col0 = n0 + c * 32;
            if (col0 >= p.d) break;
            float x[32];
            tmem_ld32(tacc + c * 32, x);
            if (!valid) continue;
            float oh[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) oh[j] = 0.f;
            for (int h = 0; h < n_hit; ++h) {
                const int slot = static_cast<int>(p.keys[lo + h] & 0xFFFFFFFFull);
                const int t = p.rows[sc.c0 + slot];
                if (!GRPO_DCHECK(slot < p.R && t >= 0 && t < p.N, p.status)) continue;
                const float g = p.gco[t];
                float hv[32];
                decode32_f8(p.hq + static_cast<int64_t>(slot) * p.d + col0, p.e5m2 != 0, hv);
#pragma unroll
                for (int j = 0; j < 32; ++j) oh[j] = fmaf(g, hv[j], oh[j]);
            }
            float* o = out + col0;
            // the four loads of the block first (they are in flight together), then the stores
            float prev[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) prev[j] = 0.f;
            if (!first_chunk) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float q[8];
                    ld_global_v8(o + 8 * j, q);
#pragma unroll
                    for (int i = 0; i < 8; ++i) prev[8 * j + i] = q[i];
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float r[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) r[i] = f * (oh[8 * j + i] - fb * x[8 * j + i]) + prev[8 * j + i];
                st_global_v8(o + 8 * j, __float_as_uint(r[0]), __float_as_uint(r[1]), __float_as_uint(r[2]),
                             __float_as_uint(r[3]), __float_as_uint(r[4]), __float_as_uint(r[5]),
                             __float_as_uint(r[6]), __float_as_uint(r[7]));
            }
        }
    }
};

struct DwPairF8T5 : DwPairF8T {
    template <bool>
    __device__ static void mma(uint32_t st, uint32_t acc, bool first) {
        mma_fmt<true>(st, acc, first);
    }
};

// Accumulators of the pair engine: by default two 256-column buffers in tensor
// memory, used alternately so an epilogue overlaps the next item's MMAs; a
// traits class with kWideAcc uses all 512 columns as one buffer (its items are
// long enough that the epilogue's share is small).
template <class T>
struct WideAcc {
    template <class U>
    static constexpr bool get(decltype(U::kWideAcc)*) { return U::kWideAcc; }
    template <class U>
    static constexpr bool get(...) { return false; }
    static constexpr bool value = get<T>(nullptr);
};

template <class T>
__device__ __forceinline__ int acc_buf(int it) {
    return WideAcc<T>::value ? 0 : (it & 1);
}

template <class T>
__device__ __forceinline__ uint32_t acc_phase(int it) {
    return WideAcc<T>::value ? (static_cast<uint32_t>(it) & 1u) : (static_cast<uint32_t>(it >> 1) & 1u);
}

template <class T, bool kBf16>
__device__ __forceinline__ void tc_pair_body(const typename T::Params& p, const CUtensorMap& mA, const CUtensorMap& mA2,
                                             const CUtensorMap& mB) {
    extern __shared__ uint8_t smem_raw[];
    typename T::Sched sc;
    // uniform across the pair: both CTAs read the same counters
    if (!T::setup(p, sc)) return;
    const int cid = static_cast<int>(blockIdx.x) >> 1;
    const int n_pairs = static_cast<int>(gridDim.x) >> 1;
    if (cid >= sc.n_units) return;   // no work for this pair: leave before touching TMEM
    const int rank = static_cast<int>(cluster_ctarank());
    const bool leader = rank == 0;

    Smem sm = carve_smem<T::kStages, T::kStageBytes>(smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int* status = p.status;

    if (threadIdx.x == 0) {
        for (int s = 0; s < T::kStages; ++s) {
            mbar_init(&sm.full[s], 1);    // leader: its producer's expect_tx + both CTAs' bytes
            mbar_init(&sm.empty[s], 1);   // the leader's MMA commit, multicast to both CTAs
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.acc_full[b], 1);    // the leader's commit, multicast
            mbar_init(&sm.acc_empty[b], 8);   // leader: the epilogue warps of both CTAs
        }
        mbar_init(sm.drain, 1);
        *sm.abort_flag = 0;
        sm.ld_count[0] = sm.ld_count[1] = sm.ld_count[2] = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&mA);
        tma_prefetch_desc(&mA2);
        tma_prefetch_desc(&mB);
    }
    if (warp == 1) {
        tmem_alloc_pair(sm.tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *sm.tmem_slot;
    const uint32_t full0 = map_cluster(smem_u32(&sm.full[0]), 0);
    const uint32_t acc_empty0 = map_cluster(smem_u32(&sm.acc_empty[0]), 0);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            int s = 0, n_issued = 0;
            uint32_t ph = 0;
            for (int unit = cid; unit < sc.n_units; unit += n_pairs) {
                const int n_items = T::items(p, sc, unit);
                const int ks = T::ksteps(p, sc, unit);
                for (int item = 0; item < n_items; ++item) {
                    const typename T::Coord c = T::coord(p, sc, unit, item, rank);
                    const uint32_t bytes = T::tx_bytes(p, sc, c);
                    for (int k = 0; k < ks; ++k) {
                        if (!mbar_wait(&sm.empty[s], ph ^ 1u, sm.abort_flag, status)) goto producer_done;
                        if (leader) mbar_arrive_expect_tx(&sm.full[s], bytes);
                        T::load(p, sc, c, k, sm.stages + s * T::kStageBytes, full0 + 8u * s, &mA, &mA2, &mB, rank);
                        ++n_issued;
                        if (++s == T::kStages) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                }
            }
        producer_done:
            sm.ld_count[0] = n_issued;
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader only)
        if (lane == 0 && leader) {
            int s = 0, n_used = 0;
            uint32_t ph = 0;
            int it = 0;
            for (int unit = cid; unit < sc.n_units; unit += n_pairs) {
                const int n_items = T::items(p, sc, unit);
                const int ks = T::ksteps(p, sc, unit);
                for (int item = 0; item < n_items; ++item, ++it) {
                    const int b = acc_buf<T>(it);
                    const uint32_t aph = acc_phase<T>(it);
                    if (!mbar_wait(&sm.acc_empty[b], aph ^ 1u, sm.abort_flag, status)) goto mma_done;
                    tc_fence_after();
                    const uint32_t acc = tmem + b * 256;
                    for (int k = 0; k < ks; ++k) {
                        if (!mbar_wait(&sm.full[s], ph, sm.abort_flag, status)) goto mma_done;
                        ++n_used;
                        tc_fence_after();
                        T::template mma<kBf16>(smem_u32(sm.stages + s * T::kStageBytes), acc, k == 0);
                        umma_pair_commit_both(&sm.empty[s]);
                        if (++s == T::kStages) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    umma_pair_commit_both(&sm.acc_full[b]);
                }
            }
        mma_done:
            sm.ld_count[1] = n_used;
            umma_pair_commit(sm.drain);
            {
                const uint32_t a = smem_u32(sm.drain);
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(a, 0)) {
                    if (globaltimer() - t0 > kWaitTimeoutNs) {
                        atomicCAS(status, 0, GRPO_ERR_TIMEOUT);
                        break;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------ epilogue (both CTAs, own rows)
        const int row = lane + 32 * (warp & 3);
        const uint32_t tq = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        int it = 0;
        for (int unit = cid; unit < sc.n_units; unit += n_pairs) {
            const int n_items = T::items(p, sc, unit);
            typename T::Epi e;
            T::epi_begin(p, sc, unit, rank, row, e);
            for (int item = 0; item < n_items; ++item, ++it) {
                const int b = acc_buf<T>(it);
                const uint32_t aph = acc_phase<T>(it);
                if (!mbar_wait(&sm.acc_full[b], aph, sm.abort_flag, status)) goto epi_done;
                tc_fence_after();
                T::template epi_item<kBf16>(p, sc, unit, item, rank, tq + b * 256, e);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (leader)
                        mbar_arrive(&sm.acc_empty[b]);
                    else
                        mbar_arrive_cluster(acc_empty0 + 8u * b);
                }
            }
            T::epi_end(p, sc, rank, e);
        }
    epi_done:;
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    // After an abort in either CTA, the loads still in flight (both CTAs' loads
    // complete on the leader's full barriers) must land before either CTA leaves.
    // The leader reads both CTAs' counts, waits for the K-stages both issued and
    // its MMA did not consume, and tells both CTAs whether that covered every
    // issued load; only when it did not do they fall back to the fixed wait.
    cluster_sync();
    if (leader && threadIdx.x == 0) {
        const uint32_t peer_cnt = map_cluster(smem_u32(const_cast<int*>(sm.ld_count)), 1);
        const uint32_t peer_abort = map_cluster(smem_u32(const_cast<int*>(sm.abort_flag)), 1);
        const int peer_issued = static_cast<int>(ld_shared_cluster_u32(peer_cnt));
        const bool aborted = *sm.abort_flag || ld_shared_cluster_u32(peer_abort) != 0;
        int settled = 1;
        if (aborted) {
            const int issued = sm.ld_count[0], used = sm.ld_count[1];
            const int both = min(issued, peer_issued);
            settled = wait_inflight<T::kStages>(sm.full, used, both) && issued == peer_issued ? 1 : 0;
        }
        sm.ld_count[2] = settled;
        st_shared_cluster_u32(peer_cnt + 8u, static_cast<uint32_t>(settled));
    }
    // the leader's MMAs write the peer's tensor memory, and the peer's loads
    // complete on the leader's barriers: nobody leaves before both are done
    cluster_sync();
    if (!sm.ld_count[2]) abort_grace(sm.abort_flag, true);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

// ====================================================================== wait self-test
// One CTA waits on an mbarrier that nothing ever completes, through the same
// bounded wait the kernels use: it must give up after kWaitTimeoutNs and
// report GRPO_ERR_TIMEOUT instead of hanging.
__global__ void __launch_bounds__(32) k_wait_selftest(int* status, unsigned long long* waited_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const uint64_t t0 = globaltimer();
    const bool done = mbar_wait(&bar, 0, &abort_flag, status);
    const uint64_t t1 = globaltimer();
    if (threadIdx.x == 0) {
        *waited_ns = t1 - t0;
        if (done) atomicCAS(status, 0, -1);   // the phase cannot have completed
    }
}

cudaError_t launch_wait_selftest(int* status, unsigned long long* waited_ns, cudaStream_t st) {
    k_wait_selftest<<<1, 32, 0, st>>>(status, waited_ns);
    return cudaGetLastError();
}

// ====================================================================== launches

// One named kernel per traits class (the names show up in profiles).
#define GRPO_TC_KERNEL(NAME, TRAITS)                                                                           \
    template <bool kBf16>                                                                                      \
    __global__ void __launch_bounds__(kThreads, 1)                                                             \
        NAME(const __grid_constant__ TRAITS::Params p, const __grid_constant__ CUtensorMap mA,                 \
             const __grid_constant__ CUtensorMap mA2, const __grid_constant__ CUtensorMap mB) {                \
        tc_body<TRAITS, kBf16>(p, mA, mA2, mB);                                                                \
    }

GRPO_TC_KERNEL(grpo_fwd_lse_kernel, FwdT)
#undef GRPO_TC_KERNEL

#define GRPO_PAIR_KERNEL(NAME, TRAITS)                                                                         \
    template <bool kBf16>                                                                                      \
    __global__ void __launch_bounds__(kThreads, 1)                                                             \
        NAME(const __grid_constant__ TRAITS::Params p, const __grid_constant__ CUtensorMap mA,                 \
             const __grid_constant__ CUtensorMap mA2, const __grid_constant__ CUtensorMap mB) {                \
        tc_pair_body<TRAITS, kBf16>(p, mA, mA2, mB);                                                           \
    }

GRPO_PAIR_KERNEL(grpo_fwd_pair_kernel, FwdPairT)
GRPO_PAIR_KERNEL(grpo_fwd_pair_e4m3_kernel, FwdPairF8T<false>)
GRPO_PAIR_KERNEL(grpo_fwd_pair_e5m2_kernel, FwdPairF8T<true>)
GRPO_PAIR_KERNEL(grpo_dh_pair_kernel, DhPairT)
GRPO_PAIR_KERNEL(grpo_dh_pair_wide_kernel, DhPairWideT)
GRPO_PAIR_KERNEL(grpo_dw_pair_kernel, DwPairT)
GRPO_PAIR_KERNEL(grpo_dh_pair_e4m3_kernel, DhPairF8T)
GRPO_PAIR_KERNEL(grpo_dh_pair_e5m2_kernel, DhPairF8T5)
GRPO_PAIR_KERNEL(grpo_dh_pair_wide_e4m3_kernel, DhPairF8WideT)
GRPO_PAIR_KERNEL(grpo_dh_pair_wide_e5m2_kernel, DhPairF8WideT5)
GRPO_PAIR_KERNEL(grpo_dw_pair_e4m3_kernel, DwPairF8T)
GRPO_PAIR_KERNEL(grpo_dw_pair_e5m2_kernel, DwPairF8T5)
#undef GRPO_PAIR_KERNEL

// Persistent launch: one CTA per SM, in clusters of kC; the grid is capped by
// how many clusters fit on the device at once, so every CTA runs concurrently.
template <class T, int kC, class K>
static cudaError_t launch_tc(K kern, const typename T::Params& p, const CUtensorMap& a, const CUtensorMap& a2,
                             const CUtensorMap& b, int n_sm, cudaStream_t st) {
    constexpr int smem = smem_bytes<T>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = n_sm / kC;
    if (kC > 1) {
        cfg.gridDim = dim3(clusters * kC);
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) == cudaSuccess && active > 0 && active < clusters)
            clusters = active;
    }
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3(clusters * kC);
    return cudaLaunchKernelEx(&cfg, kern, p, a, a2, b);
}

cudaError_t launch_fwd_pair(const FwdParams& p, const CUtensorMap& mHp, const CUtensorMap& mHr,
                            const CUtensorMap& mW, int n_sm, bool bf16, cudaStream_t st) {
    return bf16 ? launch_tc<FwdPairT, 2>(grpo_fwd_pair_kernel<true>, p, mHp, mHr, mW, n_sm, st)
                : launch_tc<FwdPairT, 2>(grpo_fwd_pair_kernel<false>, p, mHp, mHr, mW, n_sm, st);
}

cudaError_t launch_fwd_pair_fp8(const FwdParams& p, const CUtensorMap& mHp, const CUtensorMap& mHr,
                                const CUtensorMap& mW, int n_sm, bool e5m2, cudaStream_t st) {
    return e5m2 ? launch_tc<FwdPairF8T<true>, 2>(grpo_fwd_pair_e5m2_kernel<true>, p, mHp, mHr, mW, n_sm, st)
                : launch_tc<FwdPairF8T<false>, 2>(grpo_fwd_pair_e4m3_kernel<true>, p, mHp, mHr, mW, n_sm, st);
}

cudaError_t launch_dh_pair(const ChunkParams& p, const CUtensorMap& mDS, const CUtensorMap& mWmn, int n_sm, bool bf16,
                           bool wide, cudaStream_t st) {
    if (wide)
        return bf16 ? launch_tc<DhPairWideT, 2>(grpo_dh_pair_wide_kernel<true>, p, mDS, mDS, mWmn, n_sm, st)
                    : launch_tc<DhPairWideT, 2>(grpo_dh_pair_wide_kernel<false>, p, mDS, mDS, mWmn, n_sm, st);
    return bf16 ? launch_tc<DhPairT, 2>(grpo_dh_pair_kernel<true>, p, mDS, mDS, mWmn, n_sm, st)
                : launch_tc<DhPairT, 2>(grpo_dh_pair_kernel<false>, p, mDS, mDS, mWmn, n_sm, st);
}

cudaError_t launch_dw_pair(const ChunkParams& p, const CUtensorMap& mDSmn, const CUtensorMap& mHcmn, int n_sm,
                           bool bf16, cudaStream_t st) {
    return bf16 ? launch_tc<DwPairT, 2>(grpo_dw_pair_kernel<true>, p, mDSmn, mDSmn, mHcmn, n_sm, st)
                : launch_tc<DwPairT, 2>(grpo_dw_pair_kernel<false>, p, mDSmn, mDSmn, mHcmn, n_sm, st);
}

cudaError_t launch_dh_pair_fp8(const ChunkParams& p, const CUtensorMap& mQa, const CUtensorMap& mWmn, int n_sm,
                               bool wide, cudaStream_t st) {
    if (wide)
        return p.e5m2 ? launch_tc<DhPairF8WideT5, 2>(grpo_dh_pair_wide_e5m2_kernel<true>, p, mQa, mQa, mWmn, n_sm, st)
                      : launch_tc<DhPairF8WideT, 2>(grpo_dh_pair_wide_e4m3_kernel<true>, p, mQa, mQa, mWmn, n_sm, st);
    return p.e5m2 ? launch_tc<DhPairF8T5, 2>(grpo_dh_pair_e5m2_kernel<true>, p, mQa, mQa, mWmn, n_sm, st)
                  : launch_tc<DhPairF8T, 2>(grpo_dh_pair_e4m3_kernel<true>, p, mQa, mQa, mWmn, n_sm, st);
}

cudaError_t launch_dw_pair_fp8(const ChunkParams& p, const CUtensorMap& mQbmn, const CUtensorMap& mHqmn, int n_sm,
                               cudaStream_t st) {
    return p.e5m2 ? launch_tc<DwPairF8T5, 2>(grpo_dw_pair_e5m2_kernel<true>, p, mQbmn, mQbmn, mHqmn, n_sm, st)
                  : launch_tc<DwPairF8T, 2>(grpo_dw_pair_e4m3_kernel<true>, p, mQbmn, mQbmn, mHqmn, n_sm, st);
}

cudaError_t launch_fwd(const FwdParams& p, const CUtensorMap& mHp, const CUtensorMap& mHr, const CUtensorMap& mW,
                       int n_sm, bool bf16, cudaStream_t st) {
    return bf16 ? launch_tc<FwdT, 1>(grpo_fwd_lse_kernel<true>, p, mHp, mHr, mW, n_sm, st)
                : launch_tc<FwdT, 1>(grpo_fwd_lse_kernel<false>, p, mHp, mHr, mW, n_sm, st);
}

}  // namespace grpo
