// fa_decode.cu -- decode-step attention (one query per sequence, or a few
// for speculative verify) over a paged, contiguous or ring KV cache, for
// sm_103a (GB300).
//
// One fa_decode call = two launches on the caller's stream (one for a small
// step under the cluster plan, below):
//
//   tc::fa_stream_mma_kernel<D, int8V, BI, NG, CL>   (the default path:
//                                                      BI = false, CL = false)
//       Persistent stream-K kernel.  The step's work is flattened into
//       16-token tiles ordered by (sequence, KV head [x head group], tile);
//       each warp of the grid owns an equal contiguous range of that space
//       and streams it through its own ring of shared-memory stages filled by
//       TMA (cp.async.bulk.tensor with the 128-byte swizzle for K and fp16 V;
//       cp.async.bulk for int8 V and its scales).  QK and PV run on the tensor
//       cores (mma.sync m16n8k16, fp32 accumulate) with the query heads that
//       share the KV head (up to 8, or up to 16 in two groups of 8: NG = 2)
//       as the N dimension; the online softmax sits between them in
//       registers.  At the end of each unit segment the warp writes the
//       normalised output (it covered the whole unit) or a partial
//       (O, m, l).  With BI (fa_decode_batch_invariant) the units
//       are instead cut into fixed chunks that workers take whole, so a
//       sequence's result does not depend on the rest of the batch.  With
//       CL (a small step) each (sequence, KV head) unit gets one
//       thread-block cluster whose warps split its tiles and fold their
//       partials through distributed shared memory: no merge launch.
//   tc::fa_stream_merge_kernel<D, BI>        log-sum-exp merge of the
//       partials, launched with programmatic dependent launch so its CTAs
//       start as the first kernel's leave (tc::fa_stream_merge_rows_kernel<D>,
//       a warp per row, when there are many rows).
//
//   fa_split_kernel<D, GP, int8V> + fa_merge_kernel<D>   (FA_DECODE_KERNEL=simt)
//       The CUDA-core alternative: one CTA per (split, KV head, sequence),
//       per-warp cp.async.bulk rings, fp32 FMA dots with half-warp transpose
//       reductions, a shared-memory merge of the warps and a split-count
//       merge kernel.  Kept for A/B measurement and as an independent second
//       implementation in the parity tests.
//
// The method follows the mlx-native page "flash_attn_vec_hybrid.metal":
// chunked KV walk with split-K, online softmax (running M, S and the rescale
// of O), the merge of partial (O, S, M) states, and the GQA-grouped variant
// in which one K/V read serves every query head of its KV head; the tessl page
// "nn.rs" (flash_attn_decode) for the two-pass FlashDecoding split sized from
// the fixed capacity, device-side lengths and scratch that needs no zero
// fill.  Scores are kept in the base-2 domain (scale * log2 e folded into one
// multiplier), which changes no result.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <type_traits>
#include <utility>
#include <stdlib.h>

#include "../../include/fa_decode.h"

namespace fa {

constexpr int NWARPS = 4;             // consumer warps per CTA (each its own ring)
constexpr int STAGES = 3;             // shared-memory stages per warp
constexpr int STAGE_BYTES = 8192;     // one tile of K + V (+ scales)
constexpr int THREADS = NWARPS * 32;
constexpr unsigned long long WAIT_NS = 1000000000ull;  // ~1 s bound on any wait

__device__ unsigned int g_status;

// --------------------------------------------------------------- tile geometry
template <int D, bool VI8>
struct Geo {
    static constexpr int TILE = 2048 / D;      // tokens per tile: 16 (D=128), 8 (D=256)
    static constexpr int KH = TILE / 2;        // keys per half-warp
    static constexpr int NCH = D / 128;        // 8-element chunks per lane
    static constexpr int EPL = 8 * NCH;        // head_dim elements per lane
    static constexpr int K_BYTES = TILE * D * 2;
    static constexpr int V_ROW = VI8 ? D : 2 * D;
    static constexpr int V_BYTES = TILE * V_ROW;
    static constexpr int S_ROW = VI8 ? (D / 32) * 2 : 0;
    static constexpr int S_BYTES = TILE * S_ROW;
    static_assert(K_BYTES + V_BYTES + S_BYTES <= STAGE_BYTES, "stage overflow");
    static_assert((K_BYTES % 16) == 0 && (V_BYTES % 16) == 0 && (S_BYTES % 16) == 0, "align");
};

struct Params {
    const __half *q;
    const char *k;
    const char *v;
    const char *vs;
    const int *bt;
    const int *seq_lens;
    const int *window;
    float *out;
    float *ws_o;      // [B*Hq][max_splits][D]
    float2 *ws_ml;    // [B*Hq][max_splits] (m, l), m in log2 units
    int B, Hq, Hkv, G, n_hg, hpg;
    int page_size, max_blocks, num_blocks;
    long long cap;    // tokens per sequence
    float c2;         // scale * log2(e)
    int tile;         // tokens per tile
    int tps;          // tiles per split (split kernels)
    int max_splits;
    int ring;         // contiguous ring cache: token t at row t % cap, lengths unbounded
    int tq;           // queries per sequence (multi-query decode); 1 = one
    int W;            // stream-K workers (warps) in the grid
    int U_b;          // units per sequence: kv heads x head groups
    int sh;           // heads stored per workspace slot (stream-K)
    long long *pref;  // stream-K, more than 32*SCAN_REG sequences: [B+1] flattened
                      // start tile of each sequence (last entry: all tiles)
    int cpu;          // tensor-core kernel: (query, head) columns per unit, 8 or 16
    int chunk;        // batch-invariant plan: tiles per chunk (0: stream-K plan)
    int max_chunks;   // batch-invariant plan: chunk slots per unit
    const int *slot;  // contiguous / ring caches: sequence b's cache is slot slot[b] of
                      // [n_slots][Hkv][cap][D]; NULL: slot b
    int n_slots;
    int cl_ctas;      // cluster plan: CTAs per cluster (1, 2, 4 or 8)
};

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Warp-uniform bounded wait on a stage's phase.  Returns false after ~1 s.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity)
{
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity)))
        return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 256; ++i)
            if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity)))
                return true;
        if (global_ns() - t0 > WAIT_NS)
            return false;
    }
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void flag(unsigned bit)
{
    atomicOr(&g_status, bit);
}

// --------------------------------------------------------- range and paging
// Attended key range [lo, hi) of sequence b (length clamped to capacity).
__device__ __forceinline__ void attended_range(const Params &p, int b, int &lo, int &hi,
                                               bool report)
{
    long long L = p.seq_lens[b];
    if (L < 0 || (!p.ring && L > p.cap) || L > 0x7fffffffll) {
        if (report)
            flag(FA_STATUS_LEN_CLAMPED);
        L = L < 0 ? 0 : (p.ring ? 0x7fffffffll : p.cap);
    }
    const int W = p.window ? p.window[b] : 0;
    hi = static_cast<int>(L);
    // with tq queries (the last tq tokens) the window of the first one starts
    // earliest; each query's own range is masked inside the kernel
    const int first_end = hi - (p.tq > 1 ? p.tq - 1 : 0);
    lo = (W > 0 && first_end > W) ? first_end - W : 0;
    // a ring cache holds only the last cap tokens (live length min(N, cap))
    if (p.ring && (long long)hi - p.cap > lo)
        lo = static_cast<int>(hi - p.cap);
    // a slot id that names no cache slot: nothing to attend (a zero row)
    if (p.slot) {
        const int s = p.slot[b];
        if (s < 0 || s >= p.n_slots) {
            if (report)
                flag(FA_STATUS_BAD_SLOT);
            lo = hi = 0;
        }
    }
}

// Cache slot of sequence b in a contiguous or ring cache (the slot map, or b).
__device__ __forceinline__ long long cache_slot(const Params &p, int b)
{
    return p.slot ? p.slot[b] : b;
}

template <int TILE>
__device__ __forceinline__ int tiles_in(int lo, int hi)
{
    return hi > lo ? (hi - 1) / TILE - lo / TILE + 1 : 0;
}

// Byte offset of token `tok` (a tile start) of (b, kv) in a cache whose rows
// hold `row_bytes`; -1 when the block id is out of range.
__device__ __forceinline__ long long row_offset(const Params &p, int b, int kv, int tok,
                                                int row_bytes)
{
    if (p.bt) {
        const long long blk = p.bt[(long long)b * p.max_blocks + tok / p.page_size];
        if (blk < 0 || blk >= p.num_blocks)
            return -1;
        return ((blk * p.Hkv + kv) * p.page_size + tok % p.page_size) * (long long)row_bytes;
    }
    const long long r = p.ring ? tok % p.cap : tok;
    return ((cache_slot(p, b) * p.Hkv + kv) * p.cap + r) * (long long)row_bytes;
}

// ------------------------------------------------------------- reductions
// Transpose-reduce across the 16 lanes of a half-warp: each lane starts with
// NV partial sums (index = key * GP + head); afterwards lane li holds the
// complete sums of indices li*NV/16 .. (li+1)*NV/16 - 1 (NV >= 16) or of
// index li >> (4 - log2 NV) (NV < 16).
template <int NV, int STEP>
struct HalfWarpReduce {
    __device__ __forceinline__ static void run(float *v, int li)
    {
        if constexpr (STEP < 4) {
            constexpr int mask = 8 >> STEP;
            constexpr int n = NV >> STEP;          // values still held
            if constexpr (n > 1) {
                constexpr int h = n / 2;
                const bool upper = (li & mask) != 0;
#pragma unroll
                for (int i = 0; i < h; ++i) {
                    const float send = upper ? v[i] : v[i + h];
                    const float keep = upper ? v[i + h] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
                }
            } else {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
            }
            HalfWarpReduce<NV, STEP + 1>::run(v, li);
        }
    }
};

template <int NV>
__device__ __forceinline__ int reduced_index(int li, int r)
{
    if constexpr (NV >= 16) {
        return li * (NV / 16) + r;
    } else {
        constexpr int lg = NV >= 8 ? 3 : NV >= 4 ? 2 : NV >= 2 ? 1 : 0;
        return li >> (4 - lg);
    }
}

__device__ __forceinline__ void half8_to_float(const uint4 &raw, float *f)
{
    const __half2 *h = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 x = __half22float2(h[i]);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
    }
}

// ---------------------------------------------------------------- split kernel
template <int D, int GP, bool VI8>
__global__ void __launch_bounds__(THREADS, 2) fa_split_kernel(const Params p)
{
    using Gm = Geo<D, VI8>;
    constexpr int TILE = Gm::TILE, KH = Gm::KH, NCH = Gm::NCH, EPL = Gm::EPL;
    constexpr int NV = KH * GP;
    constexpr int NVL = NV >= 16 ? NV / 16 : 1;
    constexpr int NSC = TILE * GP;                 // scores per tile
    constexpr int NR = (NSC + 31) / 32;            // scores per lane in the softmax step

    // let the merge grid launch early (it waits for this grid before reading)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int z = blockIdx.x;
    const int kv = blockIdx.y / p.n_hg;
    const int hg = blockIdx.y % p.n_hg;
    const int b = blockIdx.z;

    int lo, hi;
    attended_range(p, b, lo, hi, z == 0 && blockIdx.y == 0 && threadIdx.x == 0);
    const int nt = tiles_in<TILE>(lo, hi);
    const int n_splits = (nt + p.tps - 1) / p.tps;
    if (z >= n_splits)
        return;                                    // capacity-only split: nothing to do
    const int t_first = lo / TILE + z * p.tps;     // absolute tile index
    const int t_count = min(p.tps, nt - z * p.tps);

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    float *sbuf_all = reinterpret_cast<float *>(smem + NWARPS * STAGES * STAGE_BYTES);
    float *mw = sbuf_all + NWARPS * NSC;           // [NWARPS][GP] running max
    float *lw = mw + NWARPS * GP;                  // [NWARPS][GP] sums
    float *ow = lw + NWARPS * GP;                  // [NWARPS][GP][D] partial O
    uint64_t *bars = reinterpret_cast<uint64_t *>(ow + NWARPS * GP * D);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int hw = lane >> 4;
    const int li = lane & 15;
    float *sbuf = sbuf_all + warp * NSC;
    unsigned char *my_stages = stages + warp * STAGES * STAGE_BYTES;
    const uint32_t my_bars = smem_u32(bars + warp * STAGES);

    if (lane == 0)
        for (int s = 0; s < STAGES; ++s)
            mbar_init(my_bars + 8 * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();

    // ---- query heads of this CTA, in registers (fp32), lane's 8-element chunks
    float qf[GP][EPL];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        const int gi = hg * p.hpg + g;
        const bool live = g < p.hpg && gi < p.G;
        const __half *qrow = p.q + ((long long)b * p.Hq + kv * p.G + gi) * D;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (live)
                raw = *reinterpret_cast<const uint4 *>(qrow + c * 128 + li * 8);
            half8_to_float(raw, &qf[g][c * 8]);
        }
    }

    float acc[GP][EPL];
    float m_run[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        m_run[g] = -INFINITY;
#pragma unroll
        for (int e = 0; e < EPL; ++e)
            acc[g][e] = 0.f;
    }
    float m_mine = -INFINITY;   // running max of head (lane % GP)
    float l_lane = 0.f;         // this lane's share of the sum for head (lane % GP)

    const uint64_t policy = evict_first_policy();
    // tiles of this warp: j-th is t_first + warp + j*NWARPS
    const int n_my = t_count > warp ? (t_count - warp + NWARPS - 1) / NWARPS : 0;

    auto tile_rows = [&](int ti, int &r0, int &r1) {
        const int base = ti * TILE;
        r0 = max(lo - base, 0);
        r1 = min(hi - base, TILE);
    };

    // Issue the copies of the warp's j-th tile into stage s (lane 0 only).
    auto issue = [&](int j, int s) {
        const int ti = t_first + warp + j * NWARPS;
        int r0, r1;
        tile_rows(ti, r0, r1);
        const int tok = ti * TILE;
        const uint32_t bar = my_bars + 8 * s;
        unsigned char *st = my_stages + s * STAGE_BYTES;
        const long long ko = row_offset(p, b, kv, tok, 2 * D);
        if (ko < 0) {
            flag(FA_STATUS_BAD_BLOCK);
            mbar_expect_tx(bar, 0);   // plain arrival: the phase completes with no data
            return;
        }
        const long long vo = row_offset(p, b, kv, tok, Gm::V_ROW);
        const uint32_t kbytes = (r1 - r0) * 2 * D;
        const uint32_t vbytes = (r1 - r0) * Gm::V_ROW;
        uint32_t total = kbytes + vbytes + Gm::S_BYTES;
        mbar_expect_tx(bar, total);
        bulk_g2s(smem_u32(st + r0 * 2 * D), p.k + ko + r0 * 2 * D, kbytes, bar, policy);
        bulk_g2s(smem_u32(st + Gm::K_BYTES + r0 * Gm::V_ROW), p.v + vo + r0 * Gm::V_ROW,
                 vbytes, bar, policy);
        if constexpr (VI8) {
            const long long so = row_offset(p, b, kv, tok, Gm::S_ROW);
            bulk_g2s(smem_u32(st + Gm::K_BYTES + Gm::V_BYTES), p.vs + so, Gm::S_BYTES, bar,
                     policy);
        }
    };

    if (lane == 0)
        for (int j = 0; j < STAGES && j < n_my; ++j)
            issue(j, j);
    __syncwarp();

    int j_fail = -1;
    for (int j = 0; j < n_my; ++j) {
        const int s = j % STAGES;
        const uint32_t parity = (j / STAGES) & 1;
        if (!mbar_wait_warp(my_bars + 8 * s, parity)) {
            if (lane == 0)
                flag(FA_STATUS_WAIT_TIMEOUT);
            j_fail = j;
            break;
        }
        const int ti = t_first + warp + j * NWARPS;
        int r0, r1;
        tile_rows(ti, r0, r1);
        const bool block_ok = row_offset(p, b, kv, ti * TILE, 2) >= 0;
        const unsigned char *st = my_stages + s * STAGE_BYTES;
        const bool partial = (r0 != 0) || (r1 != TILE);

        if (block_ok) {
            // ---- QK: partial dots of this lane's chunks, GP heads x KH keys
            float part[NV];
#pragma unroll
            for (int jj = 0; jj < KH; ++jj) {
                const int t = 2 * jj + hw;
                const __half *krow = reinterpret_cast<const __half *>(st) + t * D;
                float kf[EPL];
#pragma unroll
                for (int c = 0; c < NCH; ++c)
                    half8_to_float(*reinterpret_cast<const uint4 *>(krow + c * 128 + li * 8),
                                   &kf[c * 8]);
#pragma unroll
                for (int g = 0; g < GP; ++g) {
                    float sacc = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e)
                        sacc = fmaf(qf[g][e], kf[e], sacc);
                    part[jj * GP + g] = sacc;
                }
            }
            HalfWarpReduce<NV, 0>::run(part, li);
#pragma unroll
            for (int r = 0; r < NVL; ++r) {
                const int idx = reduced_index<NV>(li, r);
                const int t = 2 * (idx / GP) + hw;
                float sv = part[r] * p.c2;
                if (partial && (t < r0 || t >= r1))
                    sv = -INFINITY;
                sbuf[t * GP + idx % GP] = sv;
            }
            __syncwarp();

            // ---- online softmax: tile max per head, rescale, weights
            float sv[NR];
            float tmax = -INFINITY;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const int i = lane + 32 * r;
                sv[r] = (i < NSC) ? sbuf[i] : -INFINITY;
                tmax = fmaxf(tmax, sv[r]);
            }
#pragma unroll
            for (int mask = 16; mask >= GP; mask >>= 1)
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, mask));
            // lane holds the tile max of head (lane % GP); lane g holds head g
            bool grow = false;
            float mnew[GP];
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                mnew[g] = fmaxf(m_run[g], __shfl_sync(0xffffffffu, tmax, g));
                grow |= mnew[g] > m_run[g];
            }
            const float mnew_mine = fmaxf(m_mine, tmax);
            if (grow) {                              // identical in every lane
#pragma unroll
                for (int g = 0; g < GP; ++g) {
                    const float a = ex2(m_run[g] - mnew[g]);
#pragma unroll
                    for (int e = 0; e < EPL; ++e)
                        acc[g][e] *= a;
                    m_run[g] = mnew[g];
                }
                l_lane *= ex2(m_mine - mnew_mine);
                m_mine = mnew_mine;
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const int i = lane + 32 * r;
                if (i < NSC) {
                    const float pv = ex2(sv[r] - m_mine);
                    sbuf[i] = pv;
                    l_lane += pv;
                }
            }
            __syncwarp();

            // ---- PV: acc[g][e] += p[t][g] * V[t][e] over this half-warp's keys
#pragma unroll
            for (int jj = 0; jj < KH; ++jj) {
                const int t = 2 * jj + hw;
                if (partial && (t < r0 || t >= r1))
                    continue;
                float pg[GP];
#pragma unroll
                for (int g = 0; g < GP; ++g)
                    pg[g] = sbuf[t * GP + g];
                if constexpr (!VI8) {
                    const __half *vrow =
                        reinterpret_cast<const __half *>(st + Gm::K_BYTES) + t * D;
                    float vf[EPL];
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        half8_to_float(
                            *reinterpret_cast<const uint4 *>(vrow + c * 128 + li * 8),
                            &vf[c * 8]);
#pragma unroll
                    for (int g = 0; g < GP; ++g)
#pragma unroll
                        for (int e = 0; e < EPL; ++e)
                            acc[g][e] = fmaf(pg[g], vf[e], acc[g][e]);
                } else {
                    const int8_t *vrow =
                        reinterpret_cast<const int8_t *>(st + Gm::K_BYTES) + t * D;
                    const __half *srow =
                        reinterpret_cast<const __half *>(st + Gm::K_BYTES + Gm::V_BYTES) +
                        t * (D / 32);
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        const float sc = __half2float(srow[c * 4 + li / 4]);
                        const uint2 raw =
                            *reinterpret_cast<const uint2 *>(vrow + c * 128 + li * 8);
                        const int8_t *cb = reinterpret_cast<const int8_t *>(&raw);
#pragma unroll
                        for (int g = 0; g < GP; ++g) {
                            const float ps = pg[g] * sc;
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                acc[g][c * 8 + e] =
                                    fmaf(ps, static_cast<float>(cb[e]), acc[g][c * 8 + e]);
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && j + STAGES < n_my)
            issue(j + STAGES, s);
        __syncwarp();
    }
    if (j_fail >= 0) {
        // Drain the copies still in flight into this warp's stages (each wait
        // bounded again) so none lands after the CTA exits; this split's
        // result is void and FA_STATUS_WAIT_TIMEOUT tells the host so.
        for (int jj = j_fail; jj < n_my && jj < j_fail + STAGES; ++jj)
            mbar_wait_warp(my_bars + 8 * (jj % STAGES), (jj / STAGES) & 1);
    }

    // ---- warp epilogue: complete sums, combine half-warps, publish to smem
#pragma unroll
    for (int mask = 16; mask >= GP; mask >>= 1)
        l_lane += __shfl_xor_sync(0xffffffffu, l_lane, mask);
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int e = 0; e < EPL; ++e)
            acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], 16);
    if (hw == 0) {
#pragma unroll
        for (int g = 0; g < GP; ++g)
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                float4 *dst = reinterpret_cast<float4 *>(ow + (warp * GP + g) * D + c * 128 +
                                                         li * 8);
                dst[0] = make_float4(acc[g][c * 8 + 0], acc[g][c * 8 + 1], acc[g][c * 8 + 2],
                                     acc[g][c * 8 + 3]);
                dst[1] = make_float4(acc[g][c * 8 + 4], acc[g][c * 8 + 5], acc[g][c * 8 + 6],
                                     acc[g][c * 8 + 7]);
            }
    }
    if (lane < GP) {
        mw[warp * GP + lane] = m_mine;
        lw[warp * GP + lane] = l_lane;
    }
    __syncthreads();

    // ---- CTA merge of the NWARPS partial states (log-sum-exp), then write
    const int nh = min(p.hpg, p.G - hg * p.hpg);
    for (int idx = threadIdx.x; idx < nh * D; idx += THREADS) {
        const int g = idx / D;
        const int d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NWARPS; ++w)
            M = fmaxf(M, mw[w * GP + g]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NWARPS; ++w) {
                const float mwv = mw[w * GP + g];
                const float a = (mwv == -INFINITY) ? 0.f : ex2(mwv - M);
                L = fmaf(lw[w * GP + g], a, L);
                O = fmaf(ow[(w * GP + g) * D + d], a, O);
            }
        }
        const int h = kv * p.G + hg * p.hpg + g;
        const long long row = (long long)b * p.Hq + h;
        if (n_splits == 1) {
            p.out[row * D + d] = L > 0.f ? O / L : 0.f;
        } else {
            p.ws_o[(row * p.max_splits + z) * D + d] = O;
            if (d == 0)
                p.ws_ml[row * p.max_splits + z] = make_float2(M, L);
        }
    }
}

// ------------------------------------------------------ tensor-core split kernel
// The same (O, m, l) partial and log-sum-exp contract as fa_split_kernel, with
// stream-K work ranges and the two contractions on the tensor cores.  Per
// 16-key tile and per warp:
//   S[16 keys x 8 columns]   = K_tile[16 x D] . Q^T[D x 8]     (D/16 mma.m16n8k16)
//   O^T[D x 8 columns]      += V_tile^T[D x 16] . P^T[16 x 8]   (D/16 mma.m16n8k16)
// The N = 8 columns are the query heads that share the KV head (with several
// queries per sequence: the (query, head) pairs); more than 8 columns split
// into column groups, each its own unit.
// K and V tiles arrive by TMA tiled copies (cp.async.bulk.tensor, 64-column
// boxes, 128-byte swizzle), so the ldmatrix row reads are bank-conflict-free.
// P is rounded to fp16 for the PV product (accumulation stays fp32); its
// C-fragment is transposed into the B operand with movmatrix.
namespace tc {

constexpr int TILE = 16;
constexpr int GPH = 8;          // heads per unit (the mma N dimension)

// Build-time tuning (warps per CTA, stages per warp, CTAs per SM); the
// defaults are the best measured on GB300 across the decode workloads:
// head_dim 128 takes 2 CTAs x 4 warps x 3 stages (~100 KB each); head_dim 256
// with fp16 V takes 4 warps x 3 stages of 16 KB; with int8 V the per-tile
// dequantisation wants warps to switch between, so V is dequantised in place
// over the consumed K tile and the freed memory buys more warps: 8 x 2 stages
// at head_dim 256, 3 CTAs x 4 warps x 2 stages at 128.
#ifndef FA_TC_NW_128
#define FA_TC_NW_128 4
#endif
#ifndef FA_TC_STAGES_128
#define FA_TC_STAGES_128 3
#endif
#ifndef FA_TC_CTAS_128
#define FA_TC_CTAS_128 2
#endif
// head_dim 128 with int8 V: 3 CTAs x 4 warps x 2 stages of 7 KB, at most 168
// registers a thread; the 12 warps per SM measured 22-27% faster than 2 x 4 x 3
// on 16K-token steps (one and two queries), 2 x 6 x 2 as fast, 3 x 5 x 2 (128
// registers) slower
#ifndef FA_TC_NW_128_I8
#define FA_TC_NW_128_I8 4
#endif
#ifndef FA_TC_STAGES_128_I8
#define FA_TC_STAGES_128_I8 2
#endif
#ifndef FA_TC_CTAS_128_I8
#define FA_TC_CTAS_128_I8 3
#endif
#ifndef FA_TC_NW_256
#define FA_TC_NW_256 4
#endif
#ifndef FA_TC_STAGES_256
#define FA_TC_STAGES_256 3
#endif
#ifndef FA_TC_CTAS_256
#define FA_TC_CTAS_256 1
#endif
#ifndef FA_TC_NW_256_I8
#define FA_TC_NW_256_I8 8
#endif
#ifndef FA_TC_STAGES_256_I8
#define FA_TC_STAGES_256_I8 2
#endif
#ifndef FA_TC_CTAS_256_I8
#define FA_TC_CTAS_256_I8 1
#endif
// int8 V: dequantise into the stage's K region once QK has consumed it (1),
// or into a separate per-warp tile (0)
#ifndef FA_I8_INPLACE
#define FA_I8_INPLACE 1
#endif

// head_dim 256, fp16 V, two column groups per warp (query rows in shared
// memory): 5 warps x 2 stages measured 10% faster than the single-group
// kernel's 4 x 3 on 8-query decode (16 x 16K, 16 q / 8 kv heads)
#ifndef FA_TC_NW_256_NG2
#define FA_TC_NW_256_NG2 5
#endif
#ifndef FA_TC_STAGES_256_NG2
#define FA_TC_STAGES_256_NG2 2
#endif

// head_dim 256, int8 V, two column groups per warp: the most warps whose
// rings (2 stages) and query rows fit; 6 warps measured 15% faster than 5 and
// than the single-group kernel on 8-query decode (16 x 16K, 16 q / 8 kv heads)
#ifndef FA_TC_NW_256_I8_NG2
#define FA_TC_NW_256_I8_NG2 6
#endif

template <int D, bool VI8, int NG = 1>
struct Cfg {
    static constexpr bool TWO256 = D == 256 && !VI8 && NG == 2;
    static constexpr bool TWO256_I8 = D == 256 && VI8 && NG == 2;
    static constexpr int NW = D == 128 ? (VI8 ? FA_TC_NW_128_I8 : FA_TC_NW_128)
                                       : (VI8 ? (TWO256_I8 ? FA_TC_NW_256_I8_NG2 : FA_TC_NW_256_I8)
                                              : (TWO256 ? FA_TC_NW_256_NG2 : FA_TC_NW_256));
    static constexpr int STAGES =
        D == 128 ? (VI8 ? FA_TC_STAGES_128_I8 : FA_TC_STAGES_128)
                 : (VI8 ? FA_TC_STAGES_256_I8 : (TWO256 ? FA_TC_STAGES_256_NG2 : FA_TC_STAGES_256));
    static constexpr int BOXES = D / 64;                  // 64-column boxes per row
    static constexpr int BOX_BYTES = TILE * 128;          // 16 rows x 128 B
    static constexpr int T_BYTES = BOXES * BOX_BYTES;     // one fp16 tile (K, or fp16 V)
    static constexpr int V8_BYTES = TILE * D;             // int8 V tile
    static constexpr int S_BYTES = TILE * (D / 32) * 2;   // its fp16 scales
    static constexpr int V_STAGE = VI8 ? V8_BYTES + S_BYTES : T_BYTES;
    static constexpr int TX_BYTES = T_BYTES + V_STAGE;    // bytes landing per stage
    static constexpr int STAGE_BYTES = (TX_BYTES + 1023) / 1024 * 1024;
    static constexpr int CVT_BYTES = (VI8 && !FA_I8_INPLACE) ? T_BYTES : 0;   // dequantised V
    static constexpr int WARP_BYTES = STAGES * STAGE_BYTES + CVT_BYTES;
    static constexpr int RING_BYTES = NW * WARP_BYTES;
    static constexpr int SMEM = RING_BYTES + NW * STAGES * 8 + 1024;   // + barriers + alignment
    static constexpr int CTAS_PER_SM =
        D == 128 ? (VI8 ? FA_TC_CTAS_128_I8 : FA_TC_CTAS_128)
                 : (VI8 ? FA_TC_CTAS_256_I8 : FA_TC_CTAS_256);
    static_assert(CTAS_PER_SM * (SMEM + 1024) <= 228 * 1024, "shared memory per SM");
};

// Shared memory of the stream-K kernel: the rings and barriers, plus, when
// two column groups ride a warp at D=256 (QSM), each warp's 16 query rows,
// kept there instead of in registers.
template <int D, bool VI8, int NG>
struct Smem {
    static constexpr bool QSM = D == 256 && NG == 2;
    using CF = Cfg<D, VI8, NG>;
    static constexpr int Q_OFF = CF::RING_BYTES + 1024;              // after the barriers
    static constexpr int Q_WARP = 2 * GPH * D * 2;                   // 16 rows x D fp16
    static constexpr int BYTES = QSM ? Q_OFF + CF::NW * Q_WARP + 1024 : CF::SMEM;
    static_assert(CF::NW * CF::STAGES * 8 <= 1024, "barriers before Q_OFF");
    static_assert(CF::CTAS_PER_SM * (BYTES + 1024) <= 228 * 1024, "shared memory per SM");
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Four int8 codes -> two half2 of code * scale.  Each biased byte u = code +
// 128 becomes the fp16 1024 + u by placing it under the exponent byte 0x64;
// subtracting 1152 gives the code exactly, and one fp16 multiply by the scale
// rounds the product once (code * scale has at most 18 significant bits).
__device__ __forceinline__ void dequant4(uint32_t w, __half2 s2, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));   // 1152
    __half2 ha = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&a), bias), s2);
    __half2 hb = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&b), bias), s2);
    lo = *reinterpret_cast<const uint32_t *>(&ha);
    hi = *reinterpret_cast<const uint32_t *>(&hb);
}

// Shared address of 16-byte chunk `chunk` (0..D/8-1) of tile row `row` in a
// tile of BOXES swizzled 64-column boxes.
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int chunk)
{
    const int box = chunk >> 3;
    const int c = (chunk & 7) ^ (row & 7);
    return base + box * (TILE * 128) + row * 128 + c * 16;
}

// Distributed shared memory: the address of shared location `local` (an
// address in this CTA's window) in cluster CTA `rank`, and loads from it.
__device__ __forceinline__ uint32_t cl_map(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ float2 cl_ld2(uint32_t a)
{
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a)
                 : "memory");
    return v;
}
__device__ __forceinline__ float4 cl_ld4(uint32_t a)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}
// Every thread of every CTA of the cluster: writes before the barrier are
// visible to the cluster's reads after it.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Tile row coordinate (the tensor maps view K and V as [rows][D]); -1 for a
// block id out of range.
__device__ __forceinline__ long long tile_row(const Params &p, int b, int kv, int tok)
{
    if (p.bt) {
        const long long blk = p.bt[(long long)b * p.max_blocks + tok / p.page_size];
        if (blk < 0 || blk >= p.num_blocks)
            return -1;
        return (blk * p.Hkv + kv) * p.page_size + tok % p.page_size;
    }
    return (cache_slot(p, b) * p.Hkv + kv) * p.cap + (p.ring ? tok % p.cap : tok);
}

// Per-sequence walk over the flattened tile space.  Units (one KV head and
// head group of one sequence) are ordered by (sequence, unit); the tiles of
// a unit are its 16-token tiles intersecting the attended range [lo, hi).
//
// The stream-K plan charges each unit's start UNIT_COST tiles of work (the
// query load and the partial write a worker pays on entering a new unit):
// a unit takes n + UNIT_COST positions of the flattened space that workers
// split evenly, UNIT_COST empty ones then its n tiles, so a worker whose
// range crosses into a new unit gets that many fewer tiles.  Position of
// tile k of unit j of sequence b: P_b + j*(n_b + c) + c + k, with c =
// UNIT_COST (stream-K plan) or 0 (batch-invariant plan, which cuts real
// tiles).
#ifndef FA_UNIT_COST
#define FA_UNIT_COST 2
#endif
constexpr int UNIT_COST = FA_UNIT_COST;

// Flattened positions sequence b takes in the stream-K plan: its units x
// (n + UNIT_COST), none when it has no tiles.
__device__ __forceinline__ long long seq_span(const Params &p, int n)
{
    return n > 0 ? (long long)(n + UNIT_COST) * p.U_b : 0;
}

struct Walk {
    int b, j, k, n, lo, hi;   // sequence, unit in sequence, tile in unit, tiles per unit
    int c;                    // empty positions before each unit's tiles
    long long P;              // flattened position of sequence b's first unit

    __device__ __forceinline__ void load(const Params &p)
    {
        attended_range(p, b, lo, hi, false);
        n = tiles_in<TILE>(lo, hi);
    }
    // position at the first tile at or after flattened position t of
    // sequence b_ (whose first unit starts at P_)
    __device__ __forceinline__ void init(const Params &p, int b_, long long P_, long long t,
                                         int c_)
    {
        b = b_;
        P = P_;
        c = c_;
        load(p);
        const long long off = t - P;
        j = static_cast<int>(off / (n + c));
        const int r = static_cast<int>(off % (n + c));
        k = r < c ? 0 : r - c;
    }
    __device__ __forceinline__ void next(const Params &p)
    {
        if (++k < n)
            return;
        k = 0;
        if (++j < p.U_b)
            return;
        j = 0;
        do {
            if (n > 0)
                P += (long long)p.U_b * (n + c);
            ++b;
            if (b >= p.B)
                return;
            load(p);
        } while (n == 0);
    }
    __device__ __forceinline__ int tok() const { return (lo / TILE + k) * TILE; }
    __device__ __forceinline__ long long unit(const Params &p) const
    {
        return (long long)b * p.U_b + j;
    }
    // flattened position of the unit's first tile, and of the current tile
    __device__ __forceinline__ long long unit_start() const
    {
        return P + (long long)j * (n + c) + c;
    }
    __device__ __forceinline__ long long pos() const { return unit_start() + k; }
};

// Warp-cooperative scan over the sequences: T = the flattened positions of
// the step (tiles plus UNIT_COST per unit); when target >= 0 also the
// sequence holding position `target` and that sequence's first position;
// when want >= 0 also sequence want's first position and tile count.
// Every lane returns the same values.
__device__ __forceinline__ long long flat_scan(const Params &p, long long target, int &b_at,
                                               long long &P_at, bool report = false,
                                               long long *pref = nullptr, int want = -1,
                                               long long *P_want = nullptr,
                                               int *n_want = nullptr)
{
    const int lane = threadIdx.x & 31;
    long long run = 0;
    b_at = -1;
    P_at = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        long long c = 0;
        int nt = 0;
        if (b < p.B) {
            int lo, hi;
            attended_range(p, b, lo, hi, report);
            nt = tiles_in<TILE>(lo, hi);
            c = seq_span(p, nt);
        }
        long long x = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off)
                x += y;
        }
        const long long excl = run + x - c;
        if (pref && b < p.B)
            pref[b] = excl;
        if (want >= b0 && want < b0 + 32) {       // warp-uniform
            *P_want = __shfl_sync(0xffffffffu, excl, want - b0);
            *n_want = __shfl_sync(0xffffffffu, nt, want - b0);
        }
        if (target >= 0 && b_at < 0) {
            const unsigned hit = __ballot_sync(0xffffffffu, b < p.B && target >= excl &&
                                                                target < excl + c);
            if (hit) {
                const int src = __ffs(hit) - 1;
                b_at = b0 + src;
                P_at = __shfl_sync(0xffffffffu, excl, src);
            }
        }
        run += __shfl_sync(0xffffffffu, x, 31);
    }
    if (pref && lane == 0)
        pref[p.B] = run;
    return run;
}

// Batch-invariant plan: each unit's tiles are cut into chunks of p.chunk
// tiles counted from its first attended tile, and workers take equal
// contiguous ranges of whole chunks in (sequence, unit, chunk) order, so what
// each chunk computes depends on its own sequence alone.  Warp-cooperative
// scan over the sequences: returns the step's chunks and, through *tiles, its
// tiles; when target >= 0 also the sequence holding flattened chunk `target`
// (b_at), that sequence's first flattened tile (P_at) and first flattened
// chunk (Pc_at).  Every lane returns the same values.
__device__ __forceinline__ long long chunk_scan(const Params &p, long long target,
                                                long long *tiles, int &b_at, long long &P_at,
                                                long long &Pc_at, bool report)
{
    const int lane = threadIdx.x & 31;
    long long run_t = 0, run_c = 0;
    b_at = -1;
    P_at = 0;
    Pc_at = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        long long ct = 0, cc = 0;
        if (b < p.B) {
            int lo, hi;
            attended_range(p, b, lo, hi, report);
            const int n = tiles_in<TILE>(lo, hi);
            ct = (long long)n * p.U_b;
            cc = (long long)((n + p.chunk - 1) / p.chunk) * p.U_b;
        }
        long long xt = ct, xc = cc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long yt = __shfl_up_sync(0xffffffffu, xt, off);
            const long long yc = __shfl_up_sync(0xffffffffu, xc, off);
            if (lane >= off) {
                xt += yt;
                xc += yc;
            }
        }
        const long long et = run_t + xt - ct, ec = run_c + xc - cc;
        if (target >= 0 && b_at < 0) {
            const unsigned hit =
                __ballot_sync(0xffffffffu, b < p.B && target >= ec && target < ec + cc);
            if (hit) {
                const int src = __ffs(hit) - 1;
                b_at = b0 + src;
                P_at = __shfl_sync(0xffffffffu, et, src);
                Pc_at = __shfl_sync(0xffffffffu, ec, src);
            }
        }
        run_t += __shfl_sync(0xffffffffu, xt, 31);
        run_c += __shfl_sync(0xffffffffu, xc, 31);
    }
    if (tiles)
        *tiles = run_t;
    return run_c;
}

// Flattened tile index of chunk `off` of sequence b (whose first tile is P).
__device__ __forceinline__ long long chunk_tile(const Params &p, int b, long long P, long long off)
{
    int lo, hi;
    attended_range(p, b, lo, hi, false);
    const int n = tiles_in<TILE>(lo, hi);
    const int nch = (n + p.chunk - 1) / p.chunk;
    const long long j = off / nch;
    return P + j * n + (off - j * nch) * p.chunk;
}

// Workers actually used for T tiles (at least MIN_TPW tiles each), and the
// worker whose contiguous range holds flattened tile t.
#ifndef FA_MIN_TPW
#define FA_MIN_TPW 1
#endif
constexpr int MIN_TPW = FA_MIN_TPW;   // fewest tiles a stream-K worker is given
constexpr int SCAN_REG = 4;     // sequences per lane kept in registers by the one-pass scan
__device__ __forceinline__ int workers_for(const Params &p, long long T)
{
    long long w = T / MIN_TPW;
    if (w < 1)
        w = 1;
    return static_cast<int>(w < p.W ? w : p.W);
}
__device__ __forceinline__ long long range_start(long long w, long long T, int We)
{
    return w * T / We;
}
__device__ __forceinline__ int worker_of(long long t, long long T, int We)
{
    return static_cast<int>(((t + 1) * We - 1) / T);
}

// Persistent stream-K split kernel on the tensor cores.  Every warp is an
// independent worker: worker w streams the flattened tiles
// [w*T/We, (w+1)*T/We) through its own TMA ring, crossing unit boundaries
// without a pause.  At the end of each unit segment it writes either the
// normalised output (the unit lies wholly in its range) or a partial
// (O, m, l) to workspace slot w + unit (unique: the workers covering
// consecutive units are non-decreasing).  The merge kernel folds the slots.
// Column c (0..cpu-1) of column group cg of KV head kv, with cpu columns per
// unit: the (query j, head h) pair x = cg*cpu + c = j*G + g (head-fastest);
// live while x < tq*G.  With one query the columns are the KV head's query
// heads.
struct Col {
    bool live;
    int j;    // query index within the sequence
    int h;    // query head
};
__device__ __forceinline__ Col column(const Params &p, int kv, int cg, int c, int cpu)
{
    const int tq = p.tq > 1 ? p.tq : 1;
    const int x = cg * cpu + c;
    Col r;
    r.live = x < tq * p.G;
    r.j = x / p.G;
    r.h = kv * p.G + x % p.G;
    return r;
}

// Keys [lo, hi) column (query j) of sequence b attends: up to and including
// its own position L - tq + j, the window counted back from there.
__device__ __forceinline__ void column_range(const Params &p, int b, int L, int j, int &lo,
                                             int &hi)
{
    const int tq = p.tq > 1 ? p.tq : 1;
    hi = max(L - (tq - 1 - j), 0);
    const int W = p.window ? p.window[b] : 0;
    lo = (W > 0 && hi > W) ? hi - W : 0;
    if (p.ring && (long long)L - p.cap > lo)
        lo = static_cast<int>(L - p.cap);
}

// BI: the batch-invariant chunk plan instead of stream-K (a separate
// instantiation, so the default kernel carries none of its code).  NG: column
// groups of 8 (query, head) columns a warp carries per K/V tile; 2 lets a
// unit hold 16 columns, so more than 8 columns per KV head read each tile
// once instead of once per group.  CL: the cluster plan for small steps --
// one thread-block cluster of p.cl_ctas CTAs per unit (1, 2, 4 or 8), the
// unit's tiles split evenly over the cluster's warps, and the warps' partials
// folded through distributed shared memory at the end, so no merge kernel
// runs.
constexpr int CL_MAX_CTAS = 8;  // the portable maximum cluster size
template <int D, bool VI8, bool BI, int NG, bool CL = false>
__global__ void __launch_bounds__(Cfg<D, VI8, NG>::NW * 32, Cfg<D, VI8, NG>::CTAS_PER_SM)
    fa_stream_mma_kernel(const Params p, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV)
{
    using C = Cfg<D, VI8, NG>;
    constexpr int STAGES = C::STAGES;
    constexpr int KS = D / 16;                       // k-steps of QK, m-tiles of PV

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g4 = lane >> 2;        // fragment row group
    const int t4 = lane & 3;         // fragment column pair
    const int w = blockIdx.x * C::NW + warp;
    // fetch the TMA descriptors while the lengths are being scanned
    if (threadIdx.x == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
        if constexpr (!VI8)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmV))
                         : "memory");
    }
    int b_at = -1;
    long long P_at = 0;
    long long T = 0, t0 = 0, t1 = 0;
    int We = 0;
    int cl_j = 0, cl_n = 0;           // cluster plan: the cluster's unit and its tiles
    if constexpr (CL) {
        // cluster plan: unit u = cluster index; worker r of the cluster's
        // R = cl_ctas x NW warps takes tiles [r*n/R, (r+1)*n/R) of it.  No
        // warp leaves early: every thread must reach the cluster barriers.
        const int cs = p.cl_ctas;
        const int u = blockIdx.x / cs;
        b_at = u / p.U_b;
        cl_j = u % p.U_b;
        int lo, hi;
        attended_range(p, b_at, lo, hi, blockIdx.x % cs == 0 && threadIdx.x == 0);
        cl_n = tiles_in<TILE>(lo, hi);
        const int R = cs * C::NW;
        const int r = (blockIdx.x % cs) * C::NW + warp;
        t0 = (long long)r * cl_n / R;
        t1 = (long long)(r + 1) * cl_n / R;
        P_at = -(long long)cl_j * cl_n;   // positions count from the unit's first tile
    } else if constexpr (BI) {
        // batch-invariant plan: whole chunks per worker; [t0, t1) is the
        // tile range of chunks [c0, c1)
        long long Pc;
        const long long Tc = chunk_scan(p, -1, &T, b_at, P_at, Pc, w == 0);
        if (Tc == 0)
            return;
        We = Tc < p.W ? static_cast<int>(Tc) : p.W;
        if (w >= We)
            return;
        const long long c0 = range_start(w, Tc, We), c1 = range_start(w + 1, Tc, We);
        chunk_scan(p, c0, nullptr, b_at, P_at, Pc, false);
        t0 = chunk_tile(p, b_at, P_at, c0 - Pc);
        if (c1 < Tc) {
            int b1;
            long long P1, Pc1;
            chunk_scan(p, c1, nullptr, b1, P1, Pc1, false);
            t1 = chunk_tile(p, b1, P1, c1 - Pc1);
        } else {
            t1 = T;
        }
    } else if (p.B <= 32 * SCAN_REG) {
        // one pass: each lane keeps the tile counts of its sequences
        // (b = lane + 32 i) in registers, then locates t0 from them
        long long c[SCAN_REG], x[SCAN_REG], base[SCAN_REG];
        long long run = 0;
        const int nblk = (p.B + 31) / 32;       // blocks of 32 sequences in use
#pragma unroll
        for (int i = 0; i < SCAN_REG; ++i) {
            const int b = lane + 32 * i;
            c[i] = 0;
            x[i] = 0;
            base[i] = run;
            if (i >= nblk)                       // warp-uniform: nothing left to scan
                continue;
            if (b < p.B) {
                int lo, hi;
                attended_range(p, b, lo, hi, w == 0);   // worker 0 reports clamped lengths
                c[i] = seq_span(p, tiles_in<TILE>(lo, hi));
            }
            x[i] = c[i];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const long long y = __shfl_up_sync(0xffffffffu, x[i], off);
                if (lane >= off)
                    x[i] += y;
            }
            run += __shfl_sync(0xffffffffu, x[i], 31);
        }
        T = run;
        if (T == 0)
            return;
        We = workers_for(p, T);
        if (w >= We)
            return;
        t0 = range_start(w, T, We);
        t1 = range_start(w + 1, T, We);
#pragma unroll
        for (int i = 0; i < SCAN_REG; ++i) {
            if (i >= nblk || b_at >= 0)
                continue;
            const long long excl = base[i] + x[i] - c[i];
            const unsigned hit =
                __ballot_sync(0xffffffffu, c[i] > 0 && t0 >= excl && t0 < excl + c[i]);
            if (hit) {
                const int src = __ffs(hit) - 1;
                b_at = 32 * i + src;
                P_at = __shfl_sync(0xffffffffu, excl, src);
            }
        }
    } else {
        // worker 0 also publishes each sequence's flattened start for the merge
        T = flat_scan(p, -1, b_at, P_at, w == 0, w == 0 ? p.pref : nullptr);
        if (T == 0)
            return;
        We = workers_for(p, T);
        if (w >= We)
            return;
        t0 = range_start(w, T, We);
        t1 = range_start(w + 1, T, We);
        flat_scan(p, t0, b_at, P_at);
    }
    // [t0, t1): this worker's flattened positions; its tiles are the ones in
    // there (the stream-K plan's unit-start positions hold none)

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::RING_BYTES);
    const uint32_t ring = smem_u32(smem) + warp * C::WARP_BYTES;
    const uint32_t cvt = ring + STAGES * C::STAGE_BYTES;     // int8 V: dequantised tile
    const uint32_t my_bars = smem_u32(bars + warp * STAGES);
    using SM = Smem<D, VI8, NG>;
    constexpr bool QSM = SM::QSM;
    const uint32_t qs = smem_u32(smem) + SM::Q_OFF + warp * SM::Q_WARP;   // QSM: query rows

    if (lane == 0)
        for (int s = 0; s < STAGES; ++s)
            mbar_init(my_bars + 8 * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();

    const uint64_t policy = evict_first_policy();
    Walk pw;                          // producer position (lane 0 issues)
    if (!CL || t1 > t0)
        pw.init(p, b_at, P_at, t0, (BI || CL) ? 0 : UNIT_COST);
    else {
        pw.b = b_at;                  // a cluster-plan warp without tiles
        pw.j = cl_j;
        pw.k = pw.n = pw.c = 0;
        pw.lo = pw.hi = 0;
        pw.P = 0;
    }
    Walk cw = pw;                     // consumer position

    auto issue = [&](int s) {
        const uint32_t bar = my_bars + 8 * s;
        const int kv = pw.j / p.n_hg;
        const long long row = tile_row(p, pw.b, kv, pw.tok());
        if (row < 0) {
            flag(FA_STATUS_BAD_BLOCK);
            mbar_expect_tx(bar, 0);
            return;
        }
        mbar_expect_tx(bar, C::TX_BYTES);
        const uint32_t st = ring + s * C::STAGE_BYTES;
#pragma unroll
        for (int bx = 0; bx < C::BOXES; ++bx) {
            tma_load_2d(st + bx * C::BOX_BYTES, &tmK, bx * 64, (int)row, bar, policy);
            if constexpr (!VI8)
                tma_load_2d(st + C::T_BYTES + bx * C::BOX_BYTES, &tmV, bx * 64, (int)row, bar,
                            policy);
        }
        if constexpr (VI8) {
            // the tile's 16 int8 rows and their scale rows are contiguous
            bulk_g2s(st + C::T_BYTES, p.v + row * D, C::V8_BYTES, bar, policy);
            bulk_g2s(st + C::T_BYTES + C::V8_BYTES, p.vs + row * (D / 32) * 2, C::S_BYTES, bar,
                     policy);
        }
    };

    // Q^T of the current unit as the QK B operand, per column group gi:
    // b0 = q[column gi*8 + g4][16ks+2t4..], b1 = +8; plus this lane's two
    // softmax columns (gi*8 + 2t4, +1) and their key ranges
    constexpr int CPU = GPH * NG;          // columns per unit
    const int tq = p.tq > 1 ? p.tq : 1;
    uint32_t qb[QSM ? 1 : NG][KS][2];
    int nh = 0;                 // live columns of the unit
    int clo[NG][2], chi[NG][2]; // key ranges of this lane's columns
    auto load_q = [&](const Walk &u) {
        const int kv = u.j / p.n_hg;
        const int cg = u.j % p.n_hg;
        nh = min(CPU, tq * p.G - cg * CPU);
        if constexpr (QSM) {
            // the unit's CPU query rows in 16-byte chunks, chunk index
            // XOR-ed with the row so that ldmatrix's 8-row reads hit 8 banks
            constexpr int CH16 = D / 8;
            for (int idx = lane; idx < CPU * CH16; idx += 32) {
                const int r = idx / CH16, ch = idx % CH16;
                const Col cq = column(p, kv, cg, r, CPU);
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (cq.live)
                    v = __ldg(reinterpret_cast<const uint4 *>(
                                  p.q + (((long long)u.b * tq + cq.j) * p.Hq + cq.h) * D) +
                              ch);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 qs + r * (D * 2) + ((ch ^ (r & 7)) * 16)),
                             "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
            }
            __syncwarp();
        }
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            if constexpr (!QSM) {
                const Col cq = column(p, kv, cg, gi * GPH + g4, CPU);
                const __half *qrow = p.q + (((long long)u.b * tq + cq.j) * p.Hq + cq.h) * D;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    qb[gi][ks][0] = cq.live ? __ldg(reinterpret_cast<const unsigned *>(
                                                  qrow + ks * 16 + 2 * t4))
                                            : 0u;
                    qb[gi][ks][1] = cq.live ? __ldg(reinterpret_cast<const unsigned *>(
                                                  qrow + ks * 16 + 8 + 2 * t4))
                                            : 0u;
                }
            }
            const Col c0 = column(p, kv, cg, gi * GPH + 2 * t4, CPU);
            const Col c1 = column(p, kv, cg, gi * GPH + 2 * t4 + 1, CPU);
            column_range(p, u.b, u.hi, c0.live ? c0.j : tq - 1, clo[gi][0], chi[gi][0]);
            column_range(p, u.b, u.hi, c1.live ? c1.j : tq - 1, clo[gi][1], chi[gi][1]);
        }
    };
    // Whether a tile remains to be issued: at head_dim 128 the producer's
    // position is checked against t1; at head_dim 256 the worker's tiles are
    // counted once up front (a walk over the units in its range) and the
    // loop runs on the count.  Both give the same tiles; each form measured
    // faster for its head_dim (the 256 kernels run at the register limit).
    constexpr bool POS_LOOP = D == 128 && !CL;
    int n_my = 0;
    if constexpr (CL) {
        n_my = static_cast<int>(t1 - t0);
    } else if constexpr (!POS_LOOP) {
        Walk e = pw;
        while (e.pos() < t1) {
            const long long us = e.unit_start();
            const long long end = us + e.n < t1 ? us + e.n : t1;
            n_my += static_cast<int>(end - e.pos());
            if (us + e.n >= t1)
                break;
            e.k = e.n - 1;          // on to the next unit
            e.next(p);
        }
    }
    int n_iss = 0;                    // tiles issued so far (tile i lands in stage i % STAGES)
    while (n_iss < STAGES && (POS_LOOP ? pw.pos() < t1 : n_iss < n_my)) {
        if (lane == 0)
            issue(n_iss);
        pw.next(p);
        ++n_iss;
    }
    __syncwarp();
    load_q(cw);
    // pull a unit's query rows into L2 when its first tile is issued, so the
    // switch to that unit does not wait on HBM (lane: column lane/4, line lane%4)
    auto prefetch_q = [&](const Walk &u) {
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            const Col cq = column(p, u.j / p.n_hg, u.j % p.n_hg, gi * GPH + (lane >> 2), CPU);
            const char *base = reinterpret_cast<const char *>(
                p.q + (((long long)u.b * tq + cq.j) * p.Hq + cq.h) * D);
            if (cq.live && (lane & 3) * 128 < D * 2)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(base + (lane & 3) * 128));
        }
    };

    float acc[NG][KS][4];
    float m[NG][2], l[NG][2];
    auto reset = [&] {
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
#pragma unroll
            for (int i = 0; i < KS; ++i)
                acc[gi][i][0] = acc[gi][i][1] = acc[gi][i][2] = acc[gi][i][3] = 0.f;
            m[gi][0] = m[gi][1] = -INFINITY;
            l[gi][0] = l[gi][1] = 0.f;
        }
    };
    reset();

    int i_fail = -1;
    int ck = 0;     // batch-invariant plan: tile within the chunk (ranges start on a chunk)
    for (int i = 0; i < (POS_LOOP ? n_iss : n_my); ++i) {
        const int s = i % STAGES;
        if (!mbar_wait_warp(my_bars + 8 * s, (i / STAGES) & 1)) {
            if (lane == 0)
                flag(FA_STATUS_WAIT_TIMEOUT);
            i_fail = i;
            break;
        }
        const int kv = cw.j / p.n_hg;
        const int base = cw.tok();
        const int r0 = max(cw.lo - base, 0);
        const int r1 = min(cw.hi - base, TILE);
        const bool block_ok = tile_row(p, cw.b, kv, base) >= 0;
        const uint32_t sK = ring + s * C::STAGE_BYTES;
        const uint32_t sV = VI8 ? (FA_I8_INPLACE ? sK : cvt) : sK + C::T_BYTES;

        // int8 V: dequantise the tile into an fp16 tile at sV (same swizzled
        // layout as a TMA-loaded one); keys outside [r0, r1) become zero rows
        auto dequant_v = [&] {
                constexpr int CPR = D / 16;               // 16-code chunks per row
                const uint32_t v8 = sK + C::T_BYTES;
                const uint32_t sc = v8 + C::V8_BYTES;
                if constexpr (NG == 1) {
                    // rows across lanes (lane keeps row lane % 16 in every
                    // chunk), chunk index rotated by the row: both the int8
                    // reads and the swizzled fp16 writes of each 8-lane phase
                    // land in 8 different bank groups.  The loads of BAT
                    // chunks go out before their conversions, so one shared
                    // memory round trip serves BAT chunks.
                    constexpr int NIT = TILE * CPR / 32;  // chunks per lane
                    constexpr int BAT = NIT < 4 ? NIT : 4;
                    const int row = lane % TILE;
                    const bool live = row >= r0 && row < r1;
#pragma unroll
                    for (int k0 = 0; k0 < NIT; k0 += BAT) {
                        uint32_t w[BAT][4];
                        unsigned short sb[BAT];
#pragma unroll
                        for (int j = 0; j < BAT; ++j) {
                            const int cc = ((lane + 32 * (k0 + j)) / TILE + row) % CPR;
                            if (live) {
                                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                             : "=r"(w[j][0]), "=r"(w[j][1]), "=r"(w[j][2]),
                                               "=r"(w[j][3])
                                             : "r"(v8 + row * D + cc * 16));
                                asm volatile("ld.shared.u16 %0, [%1];"
                                             : "=h"(sb[j])
                                             : "r"(sc + (row * (D / 32) + cc / 2) * 2));
                            }
                        }
#pragma unroll
                        for (int j = 0; j < BAT; ++j) {
                            const int cc = ((lane + 32 * (k0 + j)) / TILE + row) % CPR;
                            uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                            if (live) {
                                const __half2 s2 = __half2half2(__ushort_as_half(sb[j]));
                                dequant4(w[j][0], s2, o[0], o[1]);
                                dequant4(w[j][1], s2, o[2], o[3]);
                                dequant4(w[j][2], s2, o[4], o[5]);
                                dequant4(w[j][3], s2, o[6], o[7]);
                            }
                            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                                             swz(sV, row, 2 * cc)),
                                         "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                                         : "memory");
                            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                                             swz(sV, row, 2 * cc + 1)),
                                         "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                                         : "memory");
                        }
                    }
                } else {
                    // two column groups hold twice the accumulators: one
                    // chunk at a time (batched loads cost registers there and
                    // measured 1% slower); the same chunk layout
#pragma unroll
                    for (int kk = 0; kk < TILE * CPR / 32; ++kk) {
                        const int q = lane + 32 * kk;
                        const int row = q % TILE;
                        const int cc = (q / TILE + row) % CPR;
                        uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                        if (row >= r0 && row < r1) {
                            uint32_t w0, w1, w2, w3;
                            unsigned short sb;
                            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                         : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                                         : "r"(v8 + row * D + cc * 16));
                            asm volatile("ld.shared.u16 %0, [%1];"
                                         : "=h"(sb)
                                         : "r"(sc + (row * (D / 32) + cc / 2) * 2));
                            const __half2 s2 = __half2half2(__ushort_as_half(sb));
                            dequant4(w0, s2, o[0], o[1]);
                            dequant4(w1, s2, o[2], o[3]);
                            dequant4(w2, s2, o[4], o[5]);
                            dequant4(w3, s2, o[6], o[7]);
                        }
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                                         swz(sV, row, 2 * cc)),
                                     "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                                     : "memory");
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                                         swz(sV, row, 2 * cc + 1)),
                                     "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                                     : "memory");
                    }
                }
                __syncwarp();
        };

        if (block_ok) {
            if constexpr (VI8) {
                if constexpr (!FA_I8_INPLACE)
                    dequant_v();
            } else if (r0 != 0 || r1 != TILE) {
                // keys outside [r0, r1) hold other tokens' data: zero their V
                // rows (a 128-byte row segment per box) so 0-weights stay 0
                for (int ii = lane; ii < TILE * C::BOXES * 8; ii += 32) {
                    const int row = ii / (C::BOXES * 8);
                    if (row < r0 || row >= r1) {
                        const int rem = ii % (C::BOXES * 8);
                        const uint32_t a = sV + (rem >> 3) * C::BOX_BYTES + row * 128 +
                                           (rem & 7) * 16;
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0)
                                     : "memory");
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
            }
            // ---- S = K . Q^T per column group (rows: keys g4, g4+8; cols:
            // 2t4, 2t4+1), even and odd k-steps in two accumulators to halve
            // the mma chain; the K fragments serve every group
            float sc4[NG][4];
            {
                float sc4b[NG][4];
#pragma unroll
                for (int gi = 0; gi < NG; ++gi)
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        sc4[gi][r] = sc4b[gi][r] = 0.f;
                const int mi = lane >> 3;
                const int krow = (mi & 1) * 8 + (lane & 7);
#pragma unroll
                for (int ks = 0; ks < KS; ks += 2) {
                    uint32_t a0, a1, a2, a3, e0, e1, e2, e3;
                    ldsm_x4(swz(sK, krow, ks * 2 + (mi >> 1)), a0, a1, a2, a3);
                    ldsm_x4(swz(sK, krow, ks * 2 + 2 + (mi >> 1)), e0, e1, e2, e3);
#pragma unroll
                    for (int gi = 0; gi < NG; ++gi) {
                        uint32_t b0, b1, c0, c1;
                        if constexpr (QSM) {
                            // rows gi*8 + 0..7, chunks 2ks .. 2ks+3: the B
                            // fragments of k-steps ks and ks+1
                            const int row = gi * GPH + (lane & 7);
                            const int ch = 2 * ks + (lane >> 3);
                            ldsm_x4(qs + row * (D * 2) + ((ch ^ (row & 7)) * 16), b0, b1, c0, c1);
                        } else {
                            b0 = qb[gi][ks][0];
                            b1 = qb[gi][ks][1];
                            c0 = qb[gi][ks + 1][0];
                            c1 = qb[gi][ks + 1][1];
                        }
                        mma16816(sc4[gi], a0, a1, a2, a3, b0, b1);
                        mma16816(sc4b[gi], e0, e1, e2, e3, c0, c1);
                    }
                }
#pragma unroll
                for (int gi = 0; gi < NG; ++gi)
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        sc4[gi][r] += sc4b[gi][r];
            }
            if constexpr (VI8 && FA_I8_INPLACE) {
                __syncwarp();        // every lane's K reads are done: reuse the region
                dequant_v();
            }
            const int ka = base + g4, kb = base + g4 + 8;
            uint32_t pb0[NG], pb1[NG];
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
                float *sc = sc4[gi];
                // keys outside each column's own range (tile edges, and with
                // several queries the causal and window limits) weigh nothing
                sc[0] = (ka >= clo[gi][0] && ka < chi[gi][0]) ? sc[0] * p.c2 : -INFINITY;
                sc[1] = (ka >= clo[gi][1] && ka < chi[gi][1]) ? sc[1] * p.c2 : -INFINITY;
                sc[2] = (kb >= clo[gi][0] && kb < chi[gi][0]) ? sc[2] * p.c2 : -INFINITY;
                sc[3] = (kb >= clo[gi][1] && kb < chi[gi][1]) ? sc[3] * p.c2 : -INFINITY;
                // ---- online softmax per column (lanes sharing t4 share them)
                float x0 = fmaxf(sc[0], sc[2]);
                float x1 = fmaxf(sc[1], sc[3]);
#pragma unroll
                for (int mask = 4; mask <= 16; mask <<= 1) {
                    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, mask));
                    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, mask));
                }
                const float n0 = fmaxf(m[gi][0], x0);
                const float n1 = fmaxf(m[gi][1], x1);
                // a column with no key yet keeps max -inf: use 0 as its
                // reference so every ex2 below sees -inf (weight 0) instead
                // of -inf - -inf
                const float r0m = n0 == -INFINITY ? 0.f : n0;
                const float r1m = n1 == -INFINITY ? 0.f : n1;
                if (__any_sync(0xffffffffu, n0 > m[gi][0] || n1 > m[gi][1])) {
                    const float a0 = ex2(m[gi][0] - r0m);
                    const float a1 = ex2(m[gi][1] - r1m);
#pragma unroll
                    for (int ii = 0; ii < KS; ++ii) {
                        acc[gi][ii][0] *= a0;
                        acc[gi][ii][1] *= a1;
                        acc[gi][ii][2] *= a0;
                        acc[gi][ii][3] *= a1;
                    }
                    l[gi][0] *= a0;
                    l[gi][1] *= a1;
                    m[gi][0] = n0;
                    m[gi][1] = n1;
                }
                const float p0 = ex2(sc[0] - r0m), p1 = ex2(sc[1] - r1m);
                const float p2 = ex2(sc[2] - r0m), p3 = ex2(sc[3] - r1m);
                l[gi][0] += p0 + p2;
                l[gi][1] += p1 + p3;
                // ---- P^T as the PV B operand (keys x columns), via movmatrix
                pb0[gi] = movmatrix_t(pack_half2(p0, p1));
                pb1[gi] = movmatrix_t(pack_half2(p2, p3));
            }
            // ---- O^T += V^T . P^T  (rows: head_dim; cols: columns); the V
            // fragments serve every group
            {
                const int mi = lane >> 3;
                const int vrow = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(swz(sV, vrow, mt * 2 + (mi & 1)), a0, a1, a2, a3);
#pragma unroll
                    for (int gi = 0; gi < NG; ++gi)
                        mma16816(acc[gi][mt], a0, a1, a2, a3, pb0[gi], pb1[gi]);
                }
            }
        }
        if constexpr (VI8 && FA_I8_INPLACE)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // before TMA refills it
        __syncwarp();
        if (POS_LOOP ? pw.pos() < t1 : i + STAGES < n_my) {   // tile i + STAGES refills stage s
            if (pw.k == 0)
                prefetch_q(pw);
            if (lane == 0)
                issue(s);
            pw.next(p);
            if constexpr (POS_LOOP)
                ++n_iss;
        }
        __syncwarp();

        if (cw.k == cw.n - 1 || i + 1 == (POS_LOOP ? n_iss : n_my) ||
            (BI && ck == p.chunk - 1)) {
            // ---- end of this worker's segment of the unit (with the
            // batch-invariant plan: of a chunk): publish it
#pragma unroll
            for (int gi = 0; gi < NG; ++gi)
#pragma unroll
                for (int mask = 4; mask <= 16; mask <<= 1) {
                    l[gi][0] += __shfl_xor_sync(0xffffffffu, l[gi][0], mask);
                    l[gi][1] += __shfl_xor_sync(0xffffffffu, l[gi][1], mask);
                }
            if constexpr (CL) {
                // cluster plan: the warp's partial waits in its drained ring,
                // [column][D] floats then [column] (m, l), for the fold below
                float *part = reinterpret_cast<float *>(smem + warp * C::WARP_BYTES);
                float2 *pml = reinterpret_cast<float2 *>(part + CPU * D);
                const int h0 = 2 * t4, h1 = h0 + 1;
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    const int d = mt * 16 + g4;
                    part[h0 * D + d] = acc[0][mt][0];
                    part[h0 * D + d + 8] = acc[0][mt][2];
                    part[h1 * D + d] = acc[0][mt][1];
                    part[h1 * D + d + 8] = acc[0][mt][3];
                }
                if (g4 == 0) {
                    pml[h0] = make_float2(m[0][0], l[0][0]);
                    pml[h1] = make_float2(m[0][1], l[0][1]);
                }
                continue;        // the warp's last tile: its range lies in one unit
            }
            bool whole;          // the segment is the whole unit: normalised output
            long long slot;      // else its partial's workspace slot
            if constexpr (BI) {
                whole = cw.n <= p.chunk;
                slot = cw.unit(p) * p.max_chunks + cw.k / p.chunk;
            } else {
                const long long us = cw.unit_start();
                const int wf = worker_of(us, T, We);
                const int wl = worker_of(us + cw.n - 1, T, We);
                whole = wf == wl;
                slot = w + cw.unit(p);
            }
            const int kvu = cw.j / p.n_hg, cgu = cw.j % p.n_hg;
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
                const int h0 = gi * GPH + 2 * t4, h1 = h0 + 1;   // this lane's columns
                const Col c0 = column(p, kvu, cgu, h0, CPU), c1 = column(p, kvu, cgu, h1, CPU);
                if (whole) {
                    // the whole unit was ours: normalised output
                    const float i0 = l[gi][0] > 0.f ? 1.f / l[gi][0] : 0.f;
                    const float i1 = l[gi][1] > 0.f ? 1.f / l[gi][1] : 0.f;
                    float *o0 = p.out + (((long long)cw.b * tq + c0.j) * p.Hq + c0.h) * D;
                    float *o1 = p.out + (((long long)cw.b * tq + c1.j) * p.Hq + c1.h) * D;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        const int d = mt * 16 + g4;
                        if (c0.live) {
                            o0[d] = acc[gi][mt][0] * i0;
                            o0[d + 8] = acc[gi][mt][2] * i0;
                        }
                        if (c1.live) {
                            o1[d] = acc[gi][mt][1] * i1;
                            o1[d + 8] = acc[gi][mt][3] * i1;
                        }
                    }
                } else {
                    float *o = p.ws_o + slot * p.sh * D;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        const int d = mt * 16 + g4;
                        if (h0 < nh) {
                            o[h0 * D + d] = acc[gi][mt][0];
                            o[h0 * D + d + 8] = acc[gi][mt][2];
                        }
                        if (h1 < nh) {
                            o[h1 * D + d] = acc[gi][mt][1];
                            o[h1 * D + d + 8] = acc[gi][mt][3];
                        }
                    }
                    if (g4 == 0) {
                        if (h0 < nh)
                            p.ws_ml[slot * p.sh + h0] = make_float2(m[gi][0], l[gi][0]);
                        if (h1 < nh)
                            p.ws_ml[slot * p.sh + h1] = make_float2(m[gi][1], l[gi][1]);
                    }
                }
            }
            reset();
            if (i + 1 < (POS_LOOP ? n_iss : n_my)) {
                cw.next(p);
                if (!BI || cw.k == 0)    // a new unit (not just the next chunk)
                    load_q(cw);
            }
            ck = 0;
        } else {
            cw.next(p);
            ++ck;
        }
    }
    if (i_fail >= 0)
        for (int ii = i_fail; ii < (POS_LOOP ? n_iss : n_my) && ii < i_fail + STAGES; ++ii)
            mbar_wait_warp(my_bars + 8 * (ii % STAGES), (ii / STAGES) & 1);

    if constexpr (CL) {
        // ---- cluster plan: fold the unit's partials through distributed
        // shared memory.  A warp without tiles (or whose copies timed out)
        // leaves an empty partial: max -inf, sum 0.
        const uint32_t base = smem_u32(smem);
        if (n_my == 0 || i_fail >= 0) {
            // zero O as well, so the fold weighs every partial without a branch
            float4 *po = reinterpret_cast<float4 *>(smem + warp * C::WARP_BYTES);
            for (int x = lane; x < CPU * D / 4; x += 32)
                po[x] = make_float4(0.f, 0.f, 0.f, 0.f);
            float2 *pml = reinterpret_cast<float2 *>(po + CPU * D / 4);
            if (lane < CPU)
                pml[lane] = make_float2(-INFINITY, 0.f);
        }
        __syncwarp();
        cluster_sync();
        uint32_t rank;
        asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
        // column c of the unit: warp (c / cl_ctas) mod NW of cluster CTA
        // c % cl_ctas (one pass when the cluster has 8 warps or more, two
        // with a single 4-warp CTA)
        const int R = p.cl_ctas * C::NW;                // partials: one per warp of the cluster
        for (int c = warp * p.cl_ctas + static_cast<int>(rank); c < nh; c += R) {
            constexpr int PPL = (CL_MAX_CTAS * C::NW + 31) / 32;   // partials per lane, at most
            constexpr int EPL2 = D / 32;                // output floats per lane
            float wv[PPL], Lsum = 0.f, M = -INFINITY;
            float mv[PPL], lv[PPL];
#pragma unroll
            for (int q = 0; q < PPL; ++q) {
                const int i = lane + 32 * q;
                mv[q] = -INFINITY;
                lv[q] = 0.f;
                if (i < R) {
                    const float2 x = cl_ld2(cl_map(base + (i % C::NW) * C::WARP_BYTES +
                                                       (CPU * D + 2 * c) * 4,
                                                   i / C::NW));
                    mv[q] = x.x;
                    lv[q] = x.y;
                }
                M = fmaxf(M, mv[q]);
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
#pragma unroll
            for (int q = 0; q < PPL; ++q) {
                wv[q] = mv[q] == -INFINITY ? 0.f : ex2(mv[q] - M);
                Lsum = fmaf(lv[q], wv[q], Lsum);
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                Lsum += __shfl_xor_sync(0xffffffffu, Lsum, off);
            float o[EPL2];
#pragma unroll
            for (int e = 0; e < EPL2; ++e)
                o[e] = 0.f;
            // NB partials' loads in flight before their sums (empty partials
            // hold zeros and weigh 0): batches of 8, and one of 4 when the
            // cluster is a single 4-warp CTA.  Each batch is unrolled, so the
            // weights are picked by a select, never by a runtime index.
            auto fold = [&](const int i0, auto nb) {
                constexpr int NB = decltype(nb)::value;
                float4 x[NB][EPL2 / 4];
#pragma unroll
                for (int u = 0; u < NB; ++u) {
                    const int i = i0 + u;
                    const uint32_t src = cl_map(base + (i % C::NW) * C::WARP_BYTES +
                                                    (c * D + lane * EPL2) * 4,
                                                i / C::NW);
#pragma unroll
                    for (int e = 0; e < EPL2 / 4; ++e)
                        x[u][e] = cl_ld4(src + e * 16);
                }
#pragma unroll
                for (int u = 0; u < NB; ++u) {
                    const int i = i0 + u;
                    const float wsel = (PPL > 1 && i >= 32) ? wv[PPL - 1] : wv[0];
                    const float a = __shfl_sync(0xffffffffu, wsel, i % 32);
#pragma unroll
                    for (int e = 0; e < EPL2 / 4; ++e) {
                        o[4 * e] = fmaf(x[u][e].x, a, o[4 * e]);
                        o[4 * e + 1] = fmaf(x[u][e].y, a, o[4 * e + 1]);
                        o[4 * e + 2] = fmaf(x[u][e].z, a, o[4 * e + 2]);
                        o[4 * e + 3] = fmaf(x[u][e].w, a, o[4 * e + 3]);
                    }
                }
            };
            int i0 = 0;
            for (; i0 + 8 <= R; i0 += 8)
                fold(i0, std::integral_constant<int, 8>());
            if (i0 < R)                              // R is a multiple of 4
                fold(i0, std::integral_constant<int, 4>());
            const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
            const Col cq = column(p, cl_j / p.n_hg, cl_j % p.n_hg, c, CPU);
            float4 *dst = reinterpret_cast<float4 *>(
                p.out + (((long long)b_at * tq + cq.j) * p.Hq + cq.h) * D + lane * EPL2);
#pragma unroll
            for (int e = 0; e < EPL2; e += 4)
                dst[e / 4] = make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv,
                                         o[e + 3] * inv);
        }
        // no CTA leaves while another may still read its shared memory
        __syncwarp();
        cluster_sync();
    }
}

// Log-sum-exp merge for the stream-K kernel: one CTA of MERGE_THREADS per
// (sequence, query head) row folds the partial slots of the workers that
// covered the row's unit (or writes the zero row of an empty range).  The
// slots are spread over the threads: each thread owns one float4 column of
// D and a strided subset of the slots, so the loads of many slots are in
// flight at once; the per-slot weights ex2(m - M) are computed once into
// shared memory.
constexpr int MERGE_THREADS = 256;
// rows per SM from which the stream-K merge takes a warp per row
#ifndef FA_MERGE_WARP_ROWS_PER_SM
#define FA_MERGE_WARP_ROWS_PER_SM 4
#endif
// slots per row whose partial O the merge loads into registers up front
#ifndef FA_MERGE_REG_SLOTS_128
#define FA_MERGE_REG_SLOTS_128 32
#endif
#ifndef FA_MERGE_REG_SLOTS_256
#define FA_MERGE_REG_SLOTS_256 64
#endif
constexpr int MERGE_MAX_SLOTS = 512;   // per pass over the slots

template <int D, bool BI>
__global__ void __launch_bounds__(MERGE_THREADS) fa_stream_merge_kernel(const Params p)
{
    constexpr int CH = D / 4;                    // float4 columns
    constexpr int SG = MERGE_THREADS / CH;       // slot groups
    __shared__ float wgt[MERGE_MAX_SLOTS];
    __shared__ float red[MERGE_THREADS / 32];
    __shared__ float4 part[SG][CH];

    // row = (b * tq + query) * Hq + head; its column x = query * G + head % G
    const long long row = blockIdx.x;
    const int tq = p.tq > 1 ? p.tq : 1;
    const int b = static_cast<int>(row / ((long long)tq * p.Hq));
    const int qj = static_cast<int>((row / p.Hq) % tq);
    const int h = static_cast<int>(row % p.Hq);
    const int kv = h / p.G;
    const int x = qj * p.G + h % p.G;
    const int j = kv * p.n_hg + x / p.cpu;
    const int hh = x % p.cpu;
    const int tid = threadIdx.x;
    const int lane = tid & 31, wid = tid >> 5;

    const long long u = (long long)b * p.U_b + j;
    long long sb;    // workspace slot of the row's first partial
    int ns;          // partials to fold, in slot order
    int n;           // tiles of the row's sequence
    auto zero_row = [&] {
        if (tid < CH)
            reinterpret_cast<float4 *>(p.out + row * D)[tid] = make_float4(0.f, 0.f, 0.f, 0.f);
    };
    if constexpr (BI) {
        int lo, hi;
        attended_range(p, b, lo, hi, false);
        n = tiles_in<TILE>(lo, hi);
        if (n == 0) {
            zero_row();
            return;
        }
        // batch-invariant plan: the unit's chunks, one slot each
        ns = (n + p.chunk - 1) / p.chunk;
        if (ns == 1)
            return;                               // written by the split kernel
        asm volatile("griddepcontrol.wait;" ::: "memory");
        sb = u * p.max_chunks;
    } else {
        // T, and the flattened start and tiles of sequence b: one warp's
        // single pass over the lengths for up to 32*SCAN_REG sequences
        // (before the dependency wait, so it overlaps the split kernel's tail
        // where the CTA is resident by then), else published by the split
        // kernel's worker 0
        __shared__ long long sh_T, sh_P;
        __shared__ int sh_n;
        const bool scan_here = p.B <= 32 * SCAN_REG;
        if (scan_here) {
            if (wid == 0) {
                int b_at, nb = 0;
                long long P_at, Pb = 0;
                const long long T = flat_scan(p, -1, b_at, P_at, false, nullptr, b, &Pb, &nb);
                if (lane == 0) {
                    sh_T = T;
                    sh_P = Pb;
                    sh_n = nb;
                }
            }
            __syncthreads();
            n = sh_n;
        } else {
            int lo, hi;
            attended_range(p, b, lo, hi, false);
            n = tiles_in<TILE>(lo, hi);
        }
        if (n == 0) {                             // uniform over the CTA
            zero_row();
            return;
        }
        if (!scan_here) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            if (tid == 0) {
                sh_T = p.pref[p.B];
                sh_P = p.pref[b];
            }
            __syncthreads();
        }
        const long long T = sh_T;
        const int We = workers_for(p, T);
        const long long us = sh_P + (long long)j * (n + UNIT_COST) + UNIT_COST;   // first tile
        const int wf = worker_of(us, T, We);
        const int wl = worker_of(us + n - 1, T, We);
        if (wf == wl)
            return;                               // written by the split kernel
        if (scan_here)
            asm volatile("griddepcontrol.wait;" ::: "memory");
        sb = wf + u;
        ns = wl - wf + 1;
    }

    const int c = tid % CH;
    const int sg = tid / CH;
    // this thread's O columns of its slots (sg, sg + SG, ...): when they fit
    // in registers they are loaded before the (m, l) pairs, so both loads are
    // in flight together and the weights arrive to find them there
    constexpr int OR = (D == 128 ? FA_MERGE_REG_SLOTS_128 : FA_MERGE_REG_SLOTS_256) / SG;
    const bool in_regs = OR > 0 && ns <= SG * OR;
    float4 ov[OR > 0 ? OR : 1];
    if (in_regs) {
#pragma unroll
        for (int k = 0; k < OR; ++k) {
            const int s = sg + k * SG;
            ov[k] = s < ns ? reinterpret_cast<const float4 *>(
                                 p.ws_o + ((sb + s) * p.sh + hh) * D)[c]
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    // (m, l) of the slots: loaded once per thread (one slot per thread per
    // pass of MERGE_THREADS), reduced to M, turned into weights in shared memory
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float M = -INFINITY;
    float2 mine = make_float2(-INFINITY, 0.f);
    if (ns <= MERGE_THREADS) {
        if (tid < ns)
            mine = p.ws_ml[(sb + tid) * p.sh + hh];
        M = mine.x;
    } else {
        for (int s = tid; s < ns; s += MERGE_THREADS)
            M = fmaxf(M, p.ws_ml[(sb + s) * p.sh + hh].x);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (lane == 0)
        red[wid] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int i = 1; i < MERGE_THREADS / 32; ++i)
        M = fmaxf(M, red[i]);
    __syncthreads();

    for (int s0 = 0; s0 < ns; s0 += MERGE_MAX_SLOTS) {
        const int cnt = min(MERGE_MAX_SLOTS, ns - s0);
        float Lp = 0.f;
        for (int s = tid; s < cnt; s += MERGE_THREADS) {
            const float2 v = (ns <= MERGE_THREADS) ? mine : p.ws_ml[(sb + s0 + s) * p.sh + hh];
            const float a = (v.x == -INFINITY) ? 0.f : ex2(v.x - M);
            wgt[s] = a;
            Lp = fmaf(v.y, a, Lp);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            Lp += __shfl_xor_sync(0xffffffffu, Lp, off);
        if (lane == 0)
            red[wid] = Lp;
        __syncthreads();
#pragma unroll
        for (int i = 0; i < MERGE_THREADS / 32; ++i)
            L += red[i];
        if (in_regs) {
#pragma unroll
            for (int k = 0; k < OR; ++k) {
                const int s = sg + k * SG;
                if (s < cnt) {
                    const float a = wgt[s];
                    o.x = fmaf(ov[k].x, a, o.x);
                    o.y = fmaf(ov[k].y, a, o.y);
                    o.z = fmaf(ov[k].z, a, o.z);
                    o.w = fmaf(ov[k].w, a, o.w);
                }
            }
        } else
#pragma unroll 4
        for (int s = sg; s < cnt; s += SG) {
            const long long slot = sb + s0 + s;
            const float4 x =
                reinterpret_cast<const float4 *>(p.ws_o + (slot * p.sh + hh) * D)[c];
            const float a = wgt[s];
            o.x = fmaf(x.x, a, o.x);
            o.y = fmaf(x.y, a, o.y);
            o.z = fmaf(x.z, a, o.z);
            o.w = fmaf(x.w, a, o.w);
        }
        __syncthreads();
    }
    part[sg][c] = o;
    __syncthreads();
    if (sg == 0) {
#pragma unroll
        for (int g = 1; g < SG; ++g) {
            const float4 y = part[g][c];
            o.x += y.x;
            o.y += y.y;
            o.z += y.z;
            o.w += y.w;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        reinterpret_cast<float4 *>(p.out + row * D)[c] =
            make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
    }
}

// Warp-per-row form of the stream-K merge, for steps with many rows (the
// host picks it at four or more rows per SM): eight rows per CTA, so the
// grid runs in fewer, fuller waves and every row's length scan is one warp's
// work.  Each lane owns D/128 float4 columns of the row; the slots' weights
// are computed 32 at a time, one per lane, and broadcast by shuffles while
// the partial O columns stream in.  The fold runs in slot order.
constexpr int MERGE_ROWS_PER_CTA = 8;

template <int D>
__global__ void __launch_bounds__(MERGE_ROWS_PER_CTA * 32) fa_stream_merge_rows_kernel(
    const Params p)
{
    constexpr int CPL = D / 128;                 // float4 columns per lane
    const int lane = threadIdx.x & 31;
    const int tq = p.tq > 1 ? p.tq : 1;
    const long long rows = (long long)p.B * tq * p.Hq;
    const long long row = (long long)blockIdx.x * MERGE_ROWS_PER_CTA + (threadIdx.x >> 5);
    if (row >= rows)
        return;
    // row = (b * tq + query) * Hq + head; its column x = query * G + head % G
    const int b = static_cast<int>(row / ((long long)tq * p.Hq));
    const int qj = static_cast<int>((row / p.Hq) % tq);
    const int h = static_cast<int>(row % p.Hq);
    const int kv = h / p.G;
    const int x = qj * p.G + h % p.G;
    const int j = kv * p.n_hg + x / p.cpu;
    const int hh = x % p.cpu;
    float4 *dst = reinterpret_cast<float4 *>(p.out + row * D);

    // T, and the flattened start and tiles of sequence b (as in
    // fa_stream_merge_kernel)
    long long T = 0, P = 0;
    int n = 0;
    const bool scan_here = p.B <= 32 * SCAN_REG;
    if (scan_here) {
        int b_at;
        long long P_at;
        T = flat_scan(p, -1, b_at, P_at, false, nullptr, b, &P, &n);
    } else {
        int lo, hi;
        attended_range(p, b, lo, hi, false);
        n = tiles_in<TILE>(lo, hi);
    }
    if (n == 0) {
#pragma unroll
        for (int c = 0; c < CPL; ++c)
            dst[lane + 32 * c] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    if (!scan_here) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        T = p.pref[p.B];
        P = p.pref[b];
    }
    const int We = workers_for(p, T);
    const long long us = P + (long long)j * (n + UNIT_COST) + UNIT_COST;   // first tile
    const int wf = worker_of(us, T, We);
    const int wl = worker_of(us + n - 1, T, We);
    if (wf == wl)
        return;                                   // written by the split kernel
    if (scan_here)
        asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long sb = (long long)wf + (long long)b * p.U_b + j;
    const int ns = wl - wf + 1;
    const float2 *ml = p.ws_ml + sb * p.sh + hh;
    const float4 *po = reinterpret_cast<const float4 *>(p.ws_o + (sb * p.sh + hh) * D) + lane;
    const long long stride = (long long)p.sh * (D / 4);   // float4 per slot

    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32)
        M = fmaxf(M, ml[(long long)s * p.sh].x);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    float4 o[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c)
        o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < ns; s0 += 32) {
        const int cnt = min(32, ns - s0);
        const float2 v = lane < cnt ? ml[(long long)(s0 + lane) * p.sh]
                                    : make_float2(-INFINITY, 0.f);
        const float a = v.x == -INFINITY ? 0.f : ex2(v.x - M);
        L = fmaf(v.y, a, L);
#pragma unroll 8
        for (int k = 0; k < cnt; ++k) {
            const float ak = __shfl_sync(0xffffffffu, a, k);
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const float4 y = po[(long long)(s0 + k) * stride + 32 * c];
                o[c].x = fmaf(y.x, ak, o[c].x);
                o[c].y = fmaf(y.y, ak, o[c].y);
                o[c].z = fmaf(y.z, ak, o[c].z);
                o[c].w = fmaf(y.w, ak, o[c].w);
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        L += __shfl_xor_sync(0xffffffffu, L, off);
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c)
        dst[lane + 32 * c] = make_float4(o[c].x * inv, o[c].y * inv, o[c].z * inv, o[c].w * inv);
}

}  // namespace tc

// ---------------------------------------------------------------- merge kernel
template <int D>
__global__ void __launch_bounds__(D / 4) fa_merge_kernel(const Params p)
{
    const long long row = blockIdx.x;
    const int b = static_cast<int>(row / p.Hq);
    int lo, hi;
    attended_range(p, b, lo, hi, false);
    const int nt = hi > lo ? (hi - 1) / p.tile - lo / p.tile + 1 : 0;
    const int ns = (nt + p.tps - 1) / p.tps;
    if (ns == 1)
        return;                                   // the split kernel wrote this row
    float4 *dst = reinterpret_cast<float4 *>(p.out + row * D) + threadIdx.x;
    if (ns == 0) {
        *dst = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    // launched programmatically: wait here until the split grid's partials are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float2 *ml = p.ws_ml + row * p.max_splits;
    const float4 *po = reinterpret_cast<const float4 *>(p.ws_o + row * p.max_splits * D) +
                       threadIdx.x;
    float M = -INFINITY;
#pragma unroll 8
    for (int s = 0; s < ns; ++s)
        M = fmaxf(M, ml[s].x);
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int s = 0; s < ns; ++s) {
        const float2 v = ml[s];
        const float4 x = po[s * (D / 4)];
        const float a = (v.x == -INFINITY) ? 0.f : ex2(v.x - M);
        L = fmaf(v.y, a, L);
        o.x = fmaf(x.x, a, o.x);
        o.y = fmaf(x.y, a, o.y);
        o.z = fmaf(x.z, a, o.z);
        o.w = fmaf(x.w, a, o.w);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    *dst = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
}

// ------------------------------------------------------------ int8 V packer
// One 32-element block per warp, lane i holding element i: the block's scale
// s = fp16_rn(max|x| / 127) (the division in fp64, so the rounding is that of
// the exact quotient) and code = clamp(rint(x / s), -127, 127), 0 if s == 0.
__device__ __forceinline__ int8_t quantize32(float xv, __half &scale)
{
    float amax = fabsf(xv);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    scale = __double2half(static_cast<double>(amax) / 127.0);
    const double s = static_cast<double>(__half2float(scale));
    double qv = 0.0;
    if (s != 0.0) {
        qv = rint(static_cast<double>(xv) / s);
        qv = fmin(fmax(qv, -127.0), 127.0);
    }
    return static_cast<int8_t>(qv);
}

__global__ void fa_quantize_kernel(const float *x, long long n_blocks, int8_t *codes,
                                   __half *scales)
{
    const long long blk = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (blk >= n_blocks)
        return;
    const int lane = threadIdx.x & 31;
    __half sh;
    const int8_t c = quantize32(x[blk * 32 + lane], sh);
    codes[blk * 32 + lane] = c;
    if (lane == 0)
        scales[blk] = sh;
}

// ------------------------------------------------------------ cache append
// One CTA per (sequence, KV head): the step's K row (and V row) rounded to
// fp16, or V packed to int8 codes + per-32 scales, stored at the sequence's
// device-side position.
__global__ void fa_append_kernel(const Params p, const float *k_new, const float *v_new,
                                 __half *k_cache, void *v_cache, __half *v_scales, int D)
{
    const int b = blockIdx.x / p.Hkv;
    const int kv = blockIdx.x % p.Hkv;
    long long t = p.seq_lens[b];                // positions
    if (p.ring && t >= 0)
        t %= p.cap;
    if (t < 0 || t >= p.cap) {
        if (threadIdx.x == 0 && kv == 0)
            flag(FA_STATUS_POS_RANGE);
        return;
    }
    long long row;
    if (p.bt) {
        const long long blk = p.bt[(long long)b * p.max_blocks + t / p.page_size];
        if (blk < 0 || blk >= p.num_blocks) {
            if (threadIdx.x == 0)
                flag(FA_STATUS_BAD_BLOCK);
            return;
        }
        row = (blk * p.Hkv + kv) * p.page_size + t % p.page_size;
    } else {
        const long long sl = cache_slot(p, b);
        if (sl < 0 || sl >= p.n_slots) {       // n_slots = batch without a slot map
            if (threadIdx.x == 0 && kv == 0)
                flag(FA_STATUS_BAD_SLOT);
            return;
        }
        row = (sl * p.Hkv + kv) * p.cap + t;
    }
    const float *kr = k_new + ((long long)b * p.Hkv + kv) * D;
    const float *vr = v_new + ((long long)b * p.Hkv + kv) * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x)
        k_cache[row * D + d] = __float2half_rn(kr[d]);
    if (!v_scales) {
        __half *vc = static_cast<__half *>(v_cache);
        for (int d = threadIdx.x; d < D; d += blockDim.x)
            vc[row * D + d] = __float2half_rn(vr[d]);
    } else {
        int8_t *vc = static_cast<int8_t *>(v_cache);
        const int lane = threadIdx.x & 31;
        for (int blk = threadIdx.x >> 5; blk < D / 32; blk += blockDim.x >> 5) {
            __half sh;
            const int8_t c = quantize32(vr[blk * 32 + lane], sh);
            vc[row * D + blk * 32 + lane] = c;
            if (lane == 0)
                v_scales[row * (D / 32) + blk] = sh;
        }
    }
}

// ------------------------------------------------------------ wait self-test
// Arms a barrier that nothing will complete and waits on it with the bounded
// wait the decode kernels use: after ~1 s the wait gives up and the status
// bit is set, exactly as a copy that never lands would be reported.
__global__ void fa_wait_selftest_kernel()
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t a = smem_u32(&bar);
    if (threadIdx.x == 0)
        mbar_init(a, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();
    if (!mbar_wait_warp(a, 0) && threadIdx.x == 0)
        flag(FA_STATUS_WAIT_TIMEOUT);
}

// ------------------------------------------------------------ gather (debug)
__global__ void fa_gather_kernel(const Params p, int row_bytes, int b, int n_tokens,
                                 unsigned char *dense)
{
    const int kv = blockIdx.y;
    const int t = blockIdx.x;
    if (t >= n_tokens)
        return;
    // same page-address path as the loader: tile start, then the row within it
    const int tok = t - t % 16;
    long long off = row_offset(p, b, kv, tok, row_bytes);
    unsigned char *dst = dense + ((long long)kv * n_tokens + t) * row_bytes;
    if (off < 0) {
        if (threadIdx.x == 0)
            flag(FA_STATUS_BAD_BLOCK);
        for (int i = threadIdx.x; i < row_bytes; i += blockDim.x)
            dst[i] = 0;
        return;
    }
    off += (long long)(t - tok) * row_bytes;
    const unsigned char *src = reinterpret_cast<const unsigned char *>(p.k) + off;
    for (int i = threadIdx.x; i < row_bytes; i += blockDim.x)
        dst[i] = src[i];
}

// ================================================================ host side
static thread_local char g_err[512] = "";
static thread_local cudaEvent_t g_prof_start = nullptr;
static thread_local cudaEvent_t g_prof_end = nullptr;

static int fail(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
static int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

enum class Path { Simt, Mma };

struct Plan {
    Path path;
    int ctas;        // stream-K: persistent CTAs
    int W;           // stream-K: warps (workers)
    int sh;          // stream-K: heads per slot
    int tile;        // tokens per tile
    int gp;          // padded heads per CTA
    int hpg;         // real heads per CTA
    int n_hg;        // head groups per KV head
    int units;       // units per sequence (kv heads x head groups)
    int tps;         // tiles per split
    int max_splits;
    int chunk;       // batch-invariant plan: tiles per chunk (0: stream-K)
    int max_chunks;  // batch-invariant plan: chunk slots per unit
    int cpu;         // tensor-core kernel: columns per unit (8, or 16: two groups per warp)
};

static int next_pow2(int x)
{
    int p = 1;
    while (p < x)
        p <<= 1;
    return p;
}

// Which split kernel serves a call: the tensor-core kernel, unless
// FA_DECODE_KERNEL=simt selects the CUDA-core one (for A/B measurements; both
// compute the same result within the tolerances).  decode_impl also takes the
// CUDA-core kernel for caches of 2^31 rows or more, beyond 32-bit TMA row
// coordinates.
static Path choose_path()
{
    const char *e = getenv("FA_DECODE_KERNEL");
    if (e && !strcmp(e, "simt"))
        return Path::Simt;
    return Path::Mma;
}

// Split planner: sizes splits from batch x kv_heads x capacity so that the
// grid holds several waves of resident CTAs (the "nwg" of the pages, chosen
// here from the SM count rather than a fixed bucket).
// K/V bytes (at full capacity) from which units of 16 columns are used: four
// times GB300's 126.5 MiB L2.
constexpr double TWO_GROUP_MIN_KV_BYTES = 512.0 * (1 << 20);
// stream-K grid no larger than the capacity's tile bound allows (1), or one
// full persistent wave whatever the step (0)
#ifndef FA_GRID_CAP
#define FA_GRID_CAP 1
#endif

static Plan make_plan(Path path, int B, int Hq, int Hkv, int D, long long cap, int num_sms,
                      bool vi8, int tq = 1, int chunk = 0)
{
    Plan pl = {};
    pl.path = path;
    const int G = Hq / Hkv;
    int ctas_per_sm;
    if (path == Path::Mma) {
        pl.tile = tc::TILE;
        pl.gp = tc::GPH;
        pl.hpg = tc::GPH;
        // columns: the (query, head) pairs of one KV head, in units of 8, or
        // of 16 when there are more than 8 (a warp then carries two groups,
        // reading each K/V tile once for both).  Two groups pay off when the
        // step streams from HBM; on a step whose K/V fits in L2 the second
        // group's re-read hits L2 and the single-group units keep twice the
        // warps busy, so the choice goes by the K/V the capacity allows.
        // The batch-invariant plan keeps 8.
        const double kv_bound = (double)B * (double)cap * Hkv *
                                (2.0 * D + (vi8 ? D + D / 16.0 : 2.0 * D));
        pl.cpu = (chunk == 0 && tq * G > tc::GPH &&
                  kv_bound >= TWO_GROUP_MIN_KV_BYTES)
                     ? 2 * tc::GPH
                     : tc::GPH;
        pl.n_hg = (tq * G + pl.cpu - 1) / pl.cpu;
        pl.sh = tq * G < pl.cpu ? tq * G : pl.cpu;
        pl.units = Hkv * pl.n_hg;
        int nw, cps;
        if (D == 128) {
            nw = vi8 ? tc::Cfg<128, true>::NW : tc::Cfg<128, false>::NW;
            cps = vi8 ? tc::Cfg<128, true>::CTAS_PER_SM : tc::Cfg<128, false>::CTAS_PER_SM;
        } else if (vi8 && pl.cpu > tc::GPH) {
            nw = tc::Cfg<256, true, 2>::NW;
            cps = tc::Cfg<256, true, 2>::CTAS_PER_SM;
        } else if (vi8) {
            nw = tc::Cfg<256, true>::NW;
            cps = tc::Cfg<256, true>::CTAS_PER_SM;
        } else if (pl.cpu > tc::GPH) {
            nw = tc::Cfg<256, false, 2>::NW;          // two column groups: own warps x stages
            cps = tc::Cfg<256, false, 2>::CTAS_PER_SM;
        } else {
            nw = tc::Cfg<256, false>::NW;
            cps = tc::Cfg<256, false>::CTAS_PER_SM;
        }
        pl.ctas = (num_sms > 0 ? num_sms : 1) * cps;
        if (chunk == 0 && FA_GRID_CAP) {
            // no more workers than the capacity can give MIN_TPW positions
            // each: a step's tiles are at most batch x units x ceil(capacity / 16),
            // so a small step launches only the CTAs it can use (the device
            // plan still sizes itself from the real lengths)
            // (positions: tiles plus the unit-start cost the device plan
            // charges, so a small step still gets a worker per tile)
            const long long max_t = (long long)B * pl.units *
                                    ((cap + tc::TILE - 1) / tc::TILE + tc::UNIT_COST);
            const long long w_cap = (max_t + tc::MIN_TPW - 1) / tc::MIN_TPW;
            const long long c_cap = (w_cap + nw - 1) / nw;
            if (c_cap < pl.ctas)
                pl.ctas = static_cast<int>(c_cap > 0 ? c_cap : 1);
        }
        pl.W = pl.ctas * nw;
        pl.tps = 0;
        pl.max_splits = 0;
        if (chunk > 0) {
            // a unit holds at most ceil(cap / 16) tiles
            const long long max_tiles = (cap + tc::TILE - 1) / tc::TILE;
            pl.chunk = chunk;
            pl.max_chunks = static_cast<int>((max_tiles + chunk - 1) / chunk);
            if (pl.max_chunks < 1)
                pl.max_chunks = 1;
        }
        return pl;
    } else {
        pl.tile = 2048 / D;
        const int gpmax = D == 128 ? 4 : 2;
        if (G <= gpmax) {
            pl.gp = next_pow2(G);
            pl.hpg = G;
            pl.n_hg = 1;
        } else {
            pl.gp = gpmax;
            pl.hpg = gpmax;
            pl.n_hg = (G + gpmax - 1) / gpmax;
        }
        ctas_per_sm = 2;
    }
    const long long max_tiles = cap > 0 ? (cap + pl.tile - 1) / pl.tile : 1;
    const long long units = (long long)B * Hkv * pl.n_hg;
    const long long target = (long long)(num_sms > 0 ? num_sms : 1) * ctas_per_sm * 4 /*waves*/;
    long long tps = (units * max_tiles + target - 1) / target;
    if (tps < NWARPS)
        tps = NWARPS;
    if (tps > 256)
        tps = 256;
    pl.tps = static_cast<int>(tps);
    pl.max_splits = static_cast<int>((max_tiles + tps - 1) / tps);
    return pl;
}

// plan_workspace's answer when the bytes do not fit in a size_t
constexpr size_t WS_OVERFLOW = ~(size_t)0;

static size_t plan_workspace(const Plan &pl, int B, int Hq, int D)
{
    if (pl.path == Path::Mma && pl.chunk > 0) {
        // batch-invariant plan: one partial slot per (unit, chunk); with a
        // large capacity, short splits and many heads the product can pass
        // 2^64, and a wrapped size would let a small buffer through
        size_t n = (size_t)B;
        for (size_t f : {(size_t)pl.units, (size_t)pl.max_chunks, (size_t)pl.sh,
                         D * sizeof(float) + sizeof(float2)})
            if (__builtin_mul_overflow(n, f, &n))
                return WS_OVERFLOW;
        return n;
    }
    if (pl.path == Path::Mma) {
        // partial slots: one per (worker, unit) pair, at most W + units
        (void)Hq;
        const size_t slots = (size_t)pl.W + (size_t)B * pl.units;
        // + the per-sequence prefix published for batches the merge does not scan
        return slots * pl.sh * (D * sizeof(float) + sizeof(float2)) +
               (size_t)(B + 1) * sizeof(long long);
    }
    if (pl.max_splits <= 1)
        return 0;
    const size_t rows = (size_t)B * Hq * pl.max_splits;
    const size_t o_bytes = rows * D * sizeof(float);
    return o_bytes + rows * sizeof(float2);
}

static int device_sms(int *out)
{
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return fail(FA_ERR_CUDA, "cudaGetDevice failed");
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && cache[dev] > 0) {
        *out = cache[dev];
        return 0;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return fail(FA_ERR_CUDA, "cannot read the SM count of device %d", dev);
    if (dev < 64)
        cache[dev] = n;
    *out = n;
    return 0;
}

template <int D, int GP, bool VI8>
static size_t split_smem()
{
    constexpr int NSC = Geo<D, VI8>::TILE * GP;
    return (size_t)NWARPS * STAGES * STAGE_BYTES +
           sizeof(float) * (NWARPS * NSC + 2 * NWARPS * GP + NWARPS * GP * D) +
           sizeof(uint64_t) * NWARPS * STAGES;
}

template <int D, int GP, bool VI8>
static cudaError_t launch_split(const Params &p, dim3 grid, cudaStream_t st)
{
    const size_t smem = split_smem<D, GP, VI8>();
    static std::mutex mu;
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 64 || !done[dev]) {
            e = cudaFuncSetAttribute(fa_split_kernel<D, GP, VI8>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess)
                return e;
            if (dev < 64)
                done[dev] = true;
        }
    }
    fa_split_kernel<D, GP, VI8><<<grid, THREADS, smem, st>>>(p);
    return cudaGetLastError();
}

template <int D, bool VI8>
static cudaError_t dispatch_gp(const Params &p, int gp, dim3 grid, cudaStream_t st)
{
    switch (gp) {
    case 1: return launch_split<D, 1, VI8>(p, grid, st);
    case 2: return launch_split<D, 2, VI8>(p, grid, st);
    default:
        if constexpr (D == 128)
            return launch_split<D, 4, VI8>(p, grid, st);
        return cudaErrorInvalidValue;
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// A K or V cache viewed as a 2-D fp16 tensor [rows][D], loaded in boxes of
// 16 rows x 64 columns with the 128-byte swizzle.
static int encode_kv_map(CUtensorMap *map, const void *base, long long rows, int D)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return fail(FA_ERR_CUDA, "fa_decode: cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)tc::TILE};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FA_ERR_CUDA, "fa_decode: cuTensorMapEncodeTiled failed (%d)", (int)r);
    return 0;
}

template <int D, bool VI8, bool BI, int NG = 1>
static cudaError_t launch_mma(const Params &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                              dim3 grid, cudaStream_t st)
{
    const int smem = tc::Smem<D, VI8, NG>::BYTES;
    static std::mutex mu;
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 64 || !done[dev]) {
            e = cudaFuncSetAttribute(tc::fa_stream_mma_kernel<D, VI8, BI, NG>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess)
                return e;
            if (dev < 64)
                done[dev] = true;
        }
    }
    tc::fa_stream_mma_kernel<D, VI8, BI, NG><<<grid, tc::Cfg<D, VI8, NG>::NW * 32, smem, st>>>(
        p, tmK, tmV);
    return cudaGetLastError();
}

// Cluster plan (a cluster of 2, 4 or 8 CTAs per unit, no merge kernel): the
// most tiles per warp it takes, beyond which the stream-K plan's use of every
// SM wins over saving the merge kernel.  Measured on GB300: at head_dim 128
// it still wins with 4 tiles per warp and not with 8; at 256 with one and
// not with two.
#ifndef FA_CL_MAX_TPW_128
#define FA_CL_MAX_TPW_128 4
#endif
#ifndef FA_CL_MAX_TPW_256
#define FA_CL_MAX_TPW_256 1
#endif

// Clusters of `cs` CTAs of the cluster-plan kernel that fit on the current
// device at once (cudaOccupancyMaxActiveClusters; 0 if the query fails),
// cached per device and cluster size.
template <int D, bool VI8>
static int cluster_capacity(int cs)
{
    static std::mutex mu;
    static int cache[64][4];
    static bool done[64][4] = {};
    const int ci = cs == 1 ? 0 : cs == 2 ? 1 : cs == 4 ? 2 : 3;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && done[dev][ci])
        return cache[dev][ci];
    const int smem = tc::Smem<D, VI8, 1>::BYTES;
    int n = 0;
    if (cudaFuncSetAttribute(tc::fa_stream_mma_kernel<D, VI8, false, 1, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs * 64);
        cfg.blockDim = dim3(tc::Cfg<D, VI8>::NW * 32);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, tc::fa_stream_mma_kernel<D, VI8, false, 1, true>,
                                           &cfg) != cudaSuccess) {
            n = 0;
            cudaGetLastError();   // clear the error this refused query left (and only then)
        }
    } else {
        cudaGetLastError();       // likewise for a refused attribute
    }
    if (dev < 64) {
        cache[dev][ci] = n;
        done[dev][ci] = true;
    }
    return n;
}

template <int D, bool VI8>
static cudaError_t launch_cluster(const Params &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                  int units, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units * p.cl_ctas));
    cfg.blockDim = dim3(tc::Cfg<D, VI8>::NW * 32);
    cfg.dynamicSmemBytes = tc::Smem<D, VI8, 1>::BYTES;   // attribute set by cluster_capacity
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.cl_ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, tc::fa_stream_mma_kernel<D, VI8, false, 1, true>, p,
                                       tmK, tmV);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

static bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0)
        return false;
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

static bool aligned16(const void *x)
{
    return ((uintptr_t)x & 15u) == 0;
}

// natural alignment of an element of `bytes` bytes (a null pointer passes)
static bool aligned_to(const void *x, unsigned bytes)
{
    return ((uintptr_t)x & (bytes - 1u)) == 0;
}

// Scratch for fa_decode_noalloc: a fixed array in the module image, so that
// entry point needs no allocation.  Host code must not use the symbol's
// host-side name as a device address; noalloc_scratch() returns the real one.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

// Unique id of the calling thread's current CUDA context, 0 when none is
// current (driver entry points through the runtime, so no -lcuda).  Ids are
// never reused within a process, unlike context handles.
static unsigned long long current_ctx_id()
{
    static const auto fns = [] {
        void *cur = nullptr, *id = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &cur, 4000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            cur = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &id, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            id = nullptr;
        return std::make_pair(reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(cur),
                              reinterpret_cast<PFN_cuCtxGetId_v12000>(id));
    }();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!fns.first || !fns.second || fns.first(&ctx) != CUDA_SUCCESS || !ctx ||
        fns.second(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_noalloc_scratch in the current context, looked up once
// per context (with it current) and cached under the context's id, so a new
// context on the same device (after cudaDeviceReset, or a caller's own
// driver-API context) gets its own address.
static int noalloc_scratch(void **out)
{
    static std::mutex mu;
    constexpr int N = 64;
    static unsigned long long ids[N];
    static void *ptrs[N];
    static int used = 0, next = 0;
    unsigned long long id = current_ctx_id();
    std::lock_guard<std::mutex> lock(mu);
    if (id)
        for (int i = 0; i < used; ++i)
            if (ids[i] == id) {
                *out = ptrs[i];
                return 0;
            }
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
        int dev = -1;
        cudaGetDevice(&dev);
        return fail(FA_ERR_CUDA, "fa_decode_noalloc: cannot find the scratch array on device %d: %s",
                    dev, cudaGetErrorString(e));
    }
    if (!id)
        id = current_ctx_id();   // the lookup made the device's primary context current
    if (id) {
        const int slot = used < N ? used++ : (next++ % N);
        ids[slot] = id;
        ptrs[slot] = ptr;
    }
    *out = ptr;
    return 0;
}

}  // namespace fa

using namespace fa;

extern "C" {

FA_API const char *fa_decode_last_error(void)
{
    return g_err;
}

FA_API size_t fa_decode_workspace_size(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                       int max_kv_len, int num_sms)
{
    if (batch < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads ||
        (head_dim != 128 && head_dim != 256) || max_kv_len < 0)
        return 0;
    if (batch == 0)
        return 0;
    if (num_sms <= 0 && device_sms(&num_sms) != 0)
        return 0;
    // the caller's V type is not known here: size for whichever kernel needs more
    size_t need = 0;
    for (Path path : {Path::Simt, Path::Mma})
        for (bool vi8 : {false, true}) {
            const Plan pl = make_plan(path, batch, n_q_heads, n_kv_heads, head_dim, max_kv_len,
                                      num_sms, vi8);
            const size_t n = plan_workspace(pl, batch, n_q_heads, head_dim);
            need = n > need ? n : need;
        }
    return need;
}

static int decode_impl(const void *q, const void *k_cache, const void *v_cache,
                       const void *v_scales, const int32_t *block_table,
                       const int32_t *seq_lens, int n_q_heads, int n_kv_heads, int head_dim,
                       float scale, const int32_t *window, void *out, int batch, int page_size,
                       int max_blocks_per_seq, int num_blocks, void *workspace,
                       size_t workspace_bytes, void *stream, bool ring, int tq,
                       int chunk = 0, const int32_t *slot_ids = nullptr, int n_slots = 0);

FA_API int fa_decode(const void *q, const void *k_cache, const void *v_cache,
                     const void *v_scales, const int32_t *block_table,
                     const int32_t *seq_lens, int n_q_heads, int n_kv_heads, int head_dim,
                     float scale, const int32_t *window, void *out, int batch, int page_size,
                     int max_blocks_per_seq, int num_blocks, void *workspace,
                     size_t workspace_bytes, void *stream)
{
    return decode_impl(q, k_cache, v_cache, v_scales, block_table, seq_lens, n_q_heads,
                       n_kv_heads, head_dim, scale, window, out, batch, page_size,
                       max_blocks_per_seq, num_blocks, workspace, workspace_bytes, stream, false, 1);
}

static bool split_tokens_ok(int split_tokens)
{
    return split_tokens > 0 && split_tokens % 16 == 0 && split_tokens <= (1 << 30);
}

FA_API int fa_decode_batch_invariant(const void *q, const void *k_cache, const void *v_cache,
                                     const void *v_scales, const int32_t *block_table,
                                     const int32_t *seq_lens, int n_q_heads, int n_kv_heads,
                                     int head_dim, float scale, const int32_t *window, void *out,
                                     int batch, int page_size, int max_blocks_per_seq,
                                     int num_blocks, int split_tokens, void *workspace,
                                     size_t workspace_bytes, void *stream)
{
    g_err[0] = 0;
    if (!split_tokens_ok(split_tokens))
        return fail(FA_ERR_LAYOUT, "fa_decode_batch_invariant: split_tokens %d must be a "
                                   "positive multiple of 16", split_tokens);
    return decode_impl(q, k_cache, v_cache, v_scales, block_table, seq_lens, n_q_heads,
                       n_kv_heads, head_dim, scale, window, out, batch, page_size,
                       max_blocks_per_seq, num_blocks, workspace, workspace_bytes, stream, false, 1,
                       split_tokens / 16);
}

FA_API size_t fa_decode_batch_invariant_workspace_size(int batch, int n_q_heads, int n_kv_heads,
                                                       int head_dim, int max_kv_len,
                                                       int split_tokens)
{
    if (batch <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads ||
        (head_dim != 128 && head_dim != 256) || max_kv_len < 0 || !split_tokens_ok(split_tokens))
        return 0;
    const Plan pl = make_plan(Path::Mma, batch, n_q_heads, n_kv_heads, head_dim, max_kv_len, 1,
                              false, 1, split_tokens / 16);
    const size_t n = plan_workspace(pl, batch, n_q_heads, head_dim);
    return n == WS_OVERFLOW ? 0 : n;
}

FA_API size_t fa_decode_multi_batch_invariant_workspace_size(int batch, int n_queries,
                                                             int n_q_heads, int n_kv_heads,
                                                             int head_dim, int max_kv_len,
                                                             int split_tokens)
{
    if (n_queries <= 0 || n_queries > 256 || batch <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 ||
        n_q_heads % n_kv_heads || (head_dim != 128 && head_dim != 256) || max_kv_len < 0 ||
        !split_tokens_ok(split_tokens))
        return 0;
    const Plan pl = make_plan(Path::Mma, batch, n_q_heads, n_kv_heads, head_dim, max_kv_len, 1,
                              false, n_queries, split_tokens / 16);
    const size_t n = plan_workspace(pl, batch, n_q_heads, head_dim);
    return n == WS_OVERFLOW ? 0 : n;
}

FA_API int fa_decode_multi_batch_invariant(const void *q, const void *k_cache,
                                           const void *v_cache, const void *v_scales,
                                           const int32_t *block_table, const int32_t *seq_lens,
                                           int n_queries, int n_q_heads, int n_kv_heads,
                                           int head_dim, float scale, const int32_t *window,
                                           void *out, int batch, int page_size,
                                           int max_blocks_per_seq, int num_blocks,
                                           int split_tokens, void *workspace,
                                           size_t workspace_bytes, void *stream)
{
    g_err[0] = 0;
    if (n_queries <= 0 || n_queries > 256)
        return fail(FA_ERR_LAYOUT, "fa_decode_multi_batch_invariant: n_queries %d must be in "
                                   "[1, 256]", n_queries);
    if (!split_tokens_ok(split_tokens))
        return fail(FA_ERR_LAYOUT, "fa_decode_multi_batch_invariant: split_tokens %d must be a "
                                   "positive multiple of 16", split_tokens);
    return decode_impl(q, k_cache, v_cache, v_scales, block_table, seq_lens, n_q_heads,
                       n_kv_heads, head_dim, scale, window, out, batch, page_size,
                       max_blocks_per_seq, num_blocks, workspace, workspace_bytes, stream, false,
                       n_queries, split_tokens / 16);
}

FA_API int fa_decode_ring_batch_invariant(const void *q, const void *k_cache,
                                          const void *v_cache, const void *v_scales,
                                          const int32_t *seq_lens, int n_q_heads, int n_kv_heads,
                                          int head_dim, float scale, const int32_t *window,
                                          void *out, int batch, int capacity, int split_tokens,
                                          void *workspace, size_t workspace_bytes, void *stream)
{
    g_err[0] = 0;
    if (capacity <= 0 || capacity % 16)
        return fail(FA_ERR_LAYOUT, "fa_decode_ring_batch_invariant: capacity %d must be a "
                                   "positive multiple of 16", capacity);
    if (!split_tokens_ok(split_tokens))
        return fail(FA_ERR_LAYOUT, "fa_decode_ring_batch_invariant: split_tokens %d must be a "
                                   "positive multiple of 16", split_tokens);
    return decode_impl(q, k_cache, v_cache, v_scales, nullptr, seq_lens, n_q_heads, n_kv_heads,
                       head_dim, scale, window, out, batch, 16, capacity, 0, workspace,
                       workspace_bytes, stream, true, 1, split_tokens / 16);
}

FA_API int fa_decode_multi(const void *q, const void *k_cache, const void *v_cache,
                           const void *v_scales, const int32_t *block_table,
                           const int32_t *seq_lens, int n_queries, int n_q_heads, int n_kv_heads,
                           int head_dim, float scale, const int32_t *window, void *out, int batch,
                           int page_size, int max_blocks_per_seq, int num_blocks,
                           void *workspace, size_t workspace_bytes, void *stream)
{
    g_err[0] = 0;
    if (n_queries <= 0 || n_queries > 256)
        return fail(FA_ERR_LAYOUT, "fa_decode_multi: n_queries %d must be in [1, 256]", n_queries);
    return decode_impl(q, k_cache, v_cache, v_scales, block_table, seq_lens, n_q_heads,
                       n_kv_heads, head_dim, scale, window, out, batch, page_size,
                       max_blocks_per_seq, num_blocks, workspace, workspace_bytes, stream, false,
                       n_queries);
}

FA_API size_t fa_decode_multi_workspace_size(int batch, int n_queries, int n_q_heads,
                                             int n_kv_heads, int head_dim, int max_kv_len,
                                             int num_sms)
{
    if (n_queries <= 0 || batch < 0 || n_q_heads <= 0 || n_kv_heads <= 0 ||
        n_q_heads % n_kv_heads || (head_dim != 128 && head_dim != 256) || max_kv_len < 0)
        return 0;
    if (n_queries == 1)
        return fa_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim, max_kv_len,
                                        num_sms);
    if (batch == 0)
        return 0;
    if (num_sms <= 0 && device_sms(&num_sms) != 0)
        return 0;
    size_t need = 0;
    for (bool vi8 : {false, true}) {
        const Plan pl = make_plan(Path::Mma, batch, n_q_heads, n_kv_heads, head_dim, max_kv_len,
                                  num_sms, vi8, n_queries);
        const size_t n = plan_workspace(pl, batch, n_q_heads, head_dim);
        need = n > need ? n : need;
    }
    return need;
}

FA_API int fa_decode_ring(const void *q, const void *k_cache, const void *v_cache,
                          const void *v_scales, const int32_t *seq_lens, int n_q_heads,
                          int n_kv_heads, int head_dim, float scale, const int32_t *window,
                          void *out, int batch, int capacity, void *workspace,
                          size_t workspace_bytes, void *stream)
{
    g_err[0] = 0;
    if (capacity <= 0 || capacity % 16)
        return fail(FA_ERR_LAYOUT, "fa_decode_ring: capacity %d must be a positive multiple of 16",
                    capacity);
    return decode_impl(q, k_cache, v_cache, v_scales, nullptr, seq_lens, n_q_heads, n_kv_heads,
                       head_dim, scale, window, out, batch, 16, capacity, 0, workspace,
                       workspace_bytes, stream, true, 1);
}

FA_API int fa_decode_slots(const void *q, const void *k_cache, const void *v_cache,
                           const void *v_scales, const int32_t *slot_ids,
                           const int32_t *seq_lens, int n_q_heads, int n_kv_heads, int head_dim,
                           float scale, const int32_t *window, void *out, int batch, int n_slots,
                           int capacity, int ring, void *workspace, size_t workspace_bytes,
                           void *stream)
{
    g_err[0] = 0;
    if (!slot_ids)
        return fail(FA_ERR_NULL, "fa_decode_slots: slot_ids is required");
    if (n_slots <= 0 || capacity <= 0 || (ring && capacity % 16))
        return fail(FA_ERR_LAYOUT, "fa_decode_slots: n_slots %d and capacity %d must be positive "
                                   "(capacity a multiple of 16 for a ring)", n_slots, capacity);
    return decode_impl(q, k_cache, v_cache, v_scales, nullptr, seq_lens, n_q_heads, n_kv_heads,
                       head_dim, scale, window, out, batch, 16, capacity, 0, workspace,
                       workspace_bytes, stream, ring != 0, 1, 0, slot_ids, n_slots);
}

// The kernel path, plan and workspace need of one call: the CUDA-core path
// when FA_DECODE_KERNEL=simt or when the cache has 2^31 rows or more (TMA row
// coordinates are 32-bit), else the tensor-core kernel, which alone has the
// per-column query ranges of several queries and the chunk plan.
static int call_plan(int batch, int n_q_heads, int n_kv_heads, int D, long long cap, bool vi8,
                     bool ring, int tq, int chunk, long long kv_rows_total, int *sms, Plan *pl,
                     size_t *need)
{
    const int rc = device_sms(sms);
    if (rc)
        return rc;
    Path path = choose_path();
    if (kv_rows_total >= (1ll << 31)) {
        if (tq > 1 || chunk > 0)
            return fail(FA_ERR_LAYOUT, "fa_decode: caches of 2^31 rows or more are not "
                                       "supported with several queries or batch-invariant "
                                       "splits");
        path = Path::Simt;
    }
    if (tq > 1 || chunk > 0)
        path = Path::Mma;
    // a ring's attended range (the last cap tokens) can straddle one more tile
    *pl = make_plan(path, batch, n_q_heads, n_kv_heads, D, ring ? cap + 16 : cap, *sms, vi8, tq,
                    chunk);
    *need = plan_workspace(*pl, batch, n_q_heads, D);
    return 0;
}

static int decode_impl(const void *q, const void *k_cache, const void *v_cache,
                       const void *v_scales, const int32_t *block_table,
                       const int32_t *seq_lens, int n_q_heads, int n_kv_heads, int head_dim,
                       float scale, const int32_t *window, void *out, int batch, int page_size,
                       int max_blocks_per_seq, int num_blocks, void *workspace,
                       size_t workspace_bytes, void *stream, bool ring, int tq, int chunk,
                       const int32_t *slot_ids, int n_slots)
{
    g_err[0] = 0;
    if (!q || !k_cache || !v_cache || !seq_lens || !out)
        return fail(FA_ERR_NULL, "fa_decode: q, k_cache, v_cache, seq_lens and out are required");
    if (head_dim != 128 && head_dim != 256)
        return fail(FA_ERR_HEAD_DIM, "fa_decode: head_dim %d not supported (128 or 256)", head_dim);
    if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads ||
        n_q_heads / n_kv_heads > 64)
        return fail(FA_ERR_HEADS, "fa_decode: bad heads (q %d, kv %d)", n_q_heads, n_kv_heads);
    if (!isfinite(scale))
        return fail(FA_ERR_SCALE, "fa_decode: scale is not finite");
    if (batch < 0 || batch > 65535 || max_blocks_per_seq <= 0 || n_kv_heads > 4096)
        return fail(FA_ERR_LAYOUT, "fa_decode: bad batch %d, max_blocks_per_seq %d or kv heads %d",
                    batch, max_blocks_per_seq, n_kv_heads);
    const bool paged = block_table != nullptr;
    const bool vi8 = v_scales != nullptr;
    long long cap;
    if (paged) {
        if (page_size <= 0 || page_size % 16)
            return fail(FA_ERR_LAYOUT, "fa_decode: page_size %d must be a positive multiple of 16",
                        page_size);
        if (num_blocks <= 0)
            return fail(FA_ERR_LAYOUT, "fa_decode: num_blocks must be positive when paged");
        cap = (long long)max_blocks_per_seq * page_size;
    } else {
        cap = max_blocks_per_seq;
        if (vi8 && cap % 16)
            return fail(FA_ERR_LAYOUT,
                        "fa_decode: contiguous int8-V capacity %lld must be a multiple of 16", cap);
    }
    if (cap > (1ll << 30))
        return fail(FA_ERR_LAYOUT, "fa_decode: capacity %lld tokens too large", cap);
    if (slot_ids && (n_slots <= 0 || (double)n_slots * n_kv_heads * (double)cap > 1e15))
        return fail(FA_ERR_LAYOUT, "fa_decode: bad slot count %d for capacity %lld", n_slots, cap);
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (vi8 && !aligned16(v_scales)) || (workspace && !aligned16(workspace)))
        return fail(FA_ERR_ALIGN, "fa_decode: q, k_cache, v_cache, v_scales, out and workspace "
                                  "must be 16-byte aligned");
    if (!aligned_to(seq_lens, 4) || !aligned_to(block_table, 4) || !aligned_to(window, 4) ||
        !aligned_to(slot_ids, 4))
        return fail(FA_ERR_ALIGN, "fa_decode: seq_lens, block_table, window and slot_ids must be "
                                  "4-byte aligned");
    const int D = head_dim;
    // a contiguous or ring cache holds one slot per sequence, or n_slots
    // slots addressed through the slot map
    const long long slots = slot_ids ? (long long)n_slots : (long long)batch;
    // aliasing: out against every input range we can size
    const size_t out_bytes = (size_t)batch * tq * n_q_heads * D * sizeof(float);
    const size_t rows = paged ? (size_t)num_blocks * page_size : (size_t)slots * cap;
    const size_t kv_rows = rows * n_kv_heads;
    if (overlaps(out, out_bytes, q, (size_t)batch * tq * n_q_heads * D * 2) ||
        overlaps(out, out_bytes, k_cache, kv_rows * D * 2) ||
        overlaps(out, out_bytes, v_cache, kv_rows * D * (vi8 ? 1 : 2)) ||
        (vi8 && overlaps(out, out_bytes, v_scales, kv_rows * (D / 32) * 2)) ||
        overlaps(out, out_bytes, seq_lens, (size_t)batch * 4) ||
        (paged && overlaps(out, out_bytes, block_table, (size_t)batch * max_blocks_per_seq * 4)) ||
        (window && overlaps(out, out_bytes, window, (size_t)batch * 4)) ||
        (slot_ids && overlaps(out, out_bytes, slot_ids, (size_t)batch * 4)))
        return fail(FA_ERR_ALIAS, "fa_decode: out overlaps an input or the workspace");
    if (batch == 0)
        return 0;
    const long long kv_rows_total = paged ? (long long)num_blocks * n_kv_heads * page_size
                                          : slots * n_kv_heads * cap;
    int sms = 0;
    Plan pl;
    size_t need = 0;
    int rc = call_plan(batch, n_q_heads, n_kv_heads, D, cap, vi8, ring, tq, chunk,
                       kv_rows_total, &sms, &pl, &need);
    if (rc)
        return rc;
    if (need == WS_OVERFLOW)
        return fail(FA_ERR_WORKSPACE, "fa_decode: the workspace for these sizes exceeds 2^64 bytes");
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(FA_ERR_WORKSPACE, "fa_decode: workspace %zu bytes, need %zu", workspace_bytes,
                    need);
    if (overlaps(out, out_bytes, workspace, need))
        return fail(FA_ERR_ALIAS, "fa_decode: out overlaps the workspace");
    if (batch == 0)
        return 0;

    Params p = {};
    p.q = static_cast<const __half *>(q);
    p.k = static_cast<const char *>(k_cache);
    p.v = static_cast<const char *>(v_cache);
    p.vs = static_cast<const char *>(v_scales);
    p.bt = block_table;
    p.seq_lens = seq_lens;
    p.window = window;
    p.out = static_cast<float *>(out);
    p.ws_o = static_cast<float *>(workspace);
    p.pref = nullptr;
    if (!need) {
        p.ws_ml = nullptr;
    } else if (pl.path == Path::Mma && pl.chunk > 0) {
        const size_t slots = (size_t)batch * pl.units * pl.max_chunks;
        p.ws_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) +
                                             slots * pl.sh * D * sizeof(float));
    } else if (pl.path == Path::Mma) {
        const size_t slots = (size_t)pl.W + (size_t)batch * pl.units;
        p.ws_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) +
                                             slots * pl.sh * D * sizeof(float));
        p.pref = reinterpret_cast<long long *>(p.ws_ml + slots * pl.sh);
    } else {
        p.ws_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) +
                                             (size_t)batch * n_q_heads * pl.max_splits * D *
                                                 sizeof(float));
    }
    p.B = batch;
    p.Hq = n_q_heads;
    p.Hkv = n_kv_heads;
    p.G = n_q_heads / n_kv_heads;
    p.n_hg = pl.n_hg;
    p.hpg = pl.hpg;
    p.page_size = paged ? page_size : 16;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.cap = cap;
    p.c2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.tile = pl.tile;
    p.tps = pl.tps;
    p.max_splits = pl.max_splits;
    p.ring = ring ? 1 : 0;
    p.tq = tq;
    p.W = pl.W;
    p.U_b = n_kv_heads * pl.n_hg;
    p.sh = pl.sh;
    p.chunk = pl.chunk;
    p.max_chunks = pl.max_chunks;
    p.cpu = pl.cpu;
    p.slot = slot_ids;
    p.n_slots = static_cast<int>(slots);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 grid = pl.path == Path::Mma ? dim3(pl.ctas)
                                           : dim3(pl.max_splits, n_kv_heads * pl.n_hg, batch);
    // Small steps take the cluster plan: a cluster per unit, partials folded
    // in distributed shared memory, no merge kernel.  Only with one column
    // group, and with the largest cluster (8, 4, 2 or 1 CTAs) for which every
    // unit's cluster fits on the GPU at once and a warp gets at most
    // FA_CL_MAX_TPW_<head_dim> tiles (FA_DECODE_PLAN=streamk turns it off).
    int cluster_ctas = 0;
    if (pl.path == Path::Mma && pl.chunk == 0 && pl.cpu == tc::GPH) {
        const char *pe = getenv("FA_DECODE_PLAN");
        const long long units_all = (long long)batch * pl.units;
        const long long unit_tiles = ((ring ? cap + 16 : cap) + tc::TILE - 1) / tc::TILE;
        const int nw = D == 128 ? (vi8 ? tc::Cfg<128, true>::NW : tc::Cfg<128, false>::NW)
                                : (vi8 ? tc::Cfg<256, true>::NW : tc::Cfg<256, false>::NW);
        const long long max_tpw = D == 128 ? FA_CL_MAX_TPW_128 : FA_CL_MAX_TPW_256;
        for (int cs = tc::CL_MAX_CTAS; cs >= 1 && !(pe && !strcmp(pe, "streamk")); cs /= 2) {
            if ((unit_tiles + (long long)cs * nw - 1) / ((long long)cs * nw) > max_tpw)
                break;                       // smaller clusters give each warp more
            const int fit = D == 128 ? (vi8 ? cluster_capacity<128, true>(cs)
                                            : cluster_capacity<128, false>(cs))
                                     : (vi8 ? cluster_capacity<256, true>(cs)
                                            : cluster_capacity<256, false>(cs));
            if (units_all <= fit) {
                cluster_ctas = cs;
                break;
            }
        }
    }
    const bool cluster = cluster_ctas > 0;
    p.cl_ctas = cluster_ctas;
    cudaEvent_t prof_start = g_prof_start, prof_end = g_prof_end;
    g_prof_start = g_prof_end = nullptr;
    cudaError_t e = cudaSuccess;
    if (prof_start)
        e = cudaEventRecord(prof_start, st);
    if (e != cudaSuccess)
        return fail(FA_ERR_CUDA, "fa_decode: profile event: %s", cudaGetErrorString(e));
    if (e == cudaSuccess && pl.path == Path::Mma) {
        CUtensorMap tmK, tmV;
        const int rk = encode_kv_map(&tmK, k_cache, kv_rows_total, D);
        if (rk)
            return rk;
        if (cluster) {
            if (vi8)
                tmV = tmK;
            else if (const int rv = encode_kv_map(&tmV, v_cache, kv_rows_total, D))
                return rv;
            const int units_all = batch * pl.units;
            e = D == 128 ? (vi8 ? launch_cluster<128, true>(p, tmK, tmV, units_all, st)
                                : launch_cluster<128, false>(p, tmK, tmV, units_all, st))
                         : (vi8 ? launch_cluster<256, true>(p, tmK, tmV, units_all, st)
                                : launch_cluster<256, false>(p, tmK, tmV, units_all, st));
            if (e != cudaSuccess)
                return fail(FA_ERR_CUDA, "fa_decode: cluster launch failed: %s",
                            cudaGetErrorString(e));
            if (prof_end && (e = cudaEventRecord(prof_end, st)) != cudaSuccess)
                return fail(FA_ERR_CUDA, "fa_decode: profile event: %s", cudaGetErrorString(e));
            return 0;     // the partials were folded in the kernel: no merge
        }
        if (vi8) {
            tmV = tmK;   // unused: int8 V arrives by plain bulk copies
            if (pl.chunk > 0)
                e = D == 128 ? launch_mma<128, true, true>(p, tmK, tmV, grid, st)
                             : launch_mma<256, true, true>(p, tmK, tmV, grid, st);
            else if (pl.cpu > tc::GPH)
                e = D == 128 ? launch_mma<128, true, false, 2>(p, tmK, tmV, grid, st)
                             : launch_mma<256, true, false, 2>(p, tmK, tmV, grid, st);
            else
                e = D == 128 ? launch_mma<128, true, false>(p, tmK, tmV, grid, st)
                             : launch_mma<256, true, false>(p, tmK, tmV, grid, st);
        } else {
            const int rv = encode_kv_map(&tmV, v_cache, kv_rows_total, D);
            if (rv)
                return rv;
            if (pl.chunk > 0)
                e = D == 128 ? launch_mma<128, false, true>(p, tmK, tmV, grid, st)
                             : launch_mma<256, false, true>(p, tmK, tmV, grid, st);
            else if (pl.cpu > tc::GPH)
                e = D == 128 ? launch_mma<128, false, false, 2>(p, tmK, tmV, grid, st)
                             : launch_mma<256, false, false, 2>(p, tmK, tmV, grid, st);
            else
                e = D == 128 ? launch_mma<128, false, false>(p, tmK, tmV, grid, st)
                             : launch_mma<256, false, false>(p, tmK, tmV, grid, st);
        }
    } else if (e == cudaSuccess) {
        if (D == 128)
            e = vi8 ? dispatch_gp<128, true>(p, pl.gp, grid, st)
                    : dispatch_gp<128, false>(p, pl.gp, grid, st);
        else
            e = vi8 ? dispatch_gp<256, true>(p, pl.gp, grid, st)
                    : dispatch_gp<256, false>(p, pl.gp, grid, st);
    }
    if (e != cudaSuccess)
        return fail(FA_ERR_CUDA, "fa_decode: split launch failed: %s", cudaGetErrorString(e));
    if (prof_end && (e = cudaEventRecord(prof_end, st)) != cudaSuccess)
        return fail(FA_ERR_CUDA, "fa_decode: profile event: %s", cudaGetErrorString(e));
    {
        // programmatic dependent launch: the merge grid is scheduled while the
        // split grid drains and waits on griddepcontrol.wait for its results
        cudaLaunchConfig_t cfg = {};
        const long long rows = (long long)batch * tq * n_q_heads;
        // many rows: a warp per row, eight rows per CTA (the batch-invariant
        // plan keeps one merge form for every batch)
        const bool by_warp = pl.path == Path::Mma && pl.chunk == 0 &&
                             rows >= (long long)FA_MERGE_WARP_ROWS_PER_SM * sms;
        cfg.gridDim = by_warp ? dim3(static_cast<unsigned>(
                                    (rows + tc::MERGE_ROWS_PER_CTA - 1) / tc::MERGE_ROWS_PER_CTA))
                              : dim3(static_cast<unsigned>(rows));
        cfg.blockDim = dim3(by_warp ? tc::MERGE_ROWS_PER_CTA * 32
                                    : (pl.path == Path::Mma ? tc::MERGE_THREADS : D / 4));
        cfg.dynamicSmemBytes = 0;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = prof_end ? 0 : 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (by_warp)
            e = D == 128 ? cudaLaunchKernelEx(&cfg, tc::fa_stream_merge_rows_kernel<128>, p)
                         : cudaLaunchKernelEx(&cfg, tc::fa_stream_merge_rows_kernel<256>, p);
        else if (pl.path == Path::Mma)
            e = pl.chunk > 0
                    ? (D == 128 ? cudaLaunchKernelEx(&cfg, tc::fa_stream_merge_kernel<128, true>, p)
                                : cudaLaunchKernelEx(&cfg, tc::fa_stream_merge_kernel<256, true>, p))
                    : (D == 128 ? cudaLaunchKernelEx(&cfg, tc::fa_stream_merge_kernel<128, false>, p)
                                : cudaLaunchKernelEx(&cfg, tc::fa_stream_merge_kernel<256, false>, p));
        else
            e = D == 128 ? cudaLaunchKernelEx(&cfg, fa_merge_kernel<128>, p)
                         : cudaLaunchKernelEx(&cfg, fa_merge_kernel<256>, p);
        if (e == cudaSuccess)
            e = cudaGetLastError();
    }
    if (e != cudaSuccess)
        return fail(FA_ERR_CUDA, "fa_decode: merge launch failed: %s", cudaGetErrorString(e));
    return 0;
}

FA_API int fa_quantize_v_int8(const float *x, long long n_rows, int head_dim, int8_t *codes,
                              void *scales, void *stream)
{
    g_err[0] = 0;
    if (!x || !codes || !scales)
        return fail(FA_ERR_NULL, "fa_quantize_v_int8: null pointer");
    if (head_dim <= 0 || head_dim % 32 || n_rows < 0)
        return fail(FA_ERR_HEAD_DIM, "fa_quantize_v_int8: head_dim %d must be a positive "
                                     "multiple of 32", head_dim);
    if (!aligned_to(x, 4) || !aligned_to(scales, 2))
        return fail(FA_ERR_ALIGN, "fa_quantize_v_int8: x must be 4-byte and scales 2-byte aligned");
    const long long n_blocks = n_rows * (head_dim / 32);
    if (n_blocks == 0)
        return 0;
    const int per_cta = 8;   // warps per CTA
    const long long ctas = (n_blocks + per_cta - 1) / per_cta;
    if (ctas > 0x7fffffffll)
        return fail(FA_ERR_LAYOUT, "fa_quantize_v_int8: too many rows");
    fa_quantize_kernel<<<(unsigned)ctas, per_cta * 32, 0, static_cast<cudaStream_t>(stream)>>>(
        x, n_blocks, codes, static_cast<__half *>(scales));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(FA_ERR_CUDA, "fa_quantize_v_int8: launch failed: %s", cudaGetErrorString(e));
    return 0;
}

FA_API int fa_append_kv(const float *k_new, const float *v_new, void *k_cache, void *v_cache,
                        void *v_scales, const int32_t *block_table, const int32_t *positions,
                        int batch, int n_kv_heads, int head_dim, int page_size,
                        int max_blocks_per_seq, int num_blocks, void *stream)
{
    g_err[0] = 0;
    if (!k_new || !v_new || !k_cache || !v_cache || !positions)
        return fail(FA_ERR_NULL, "fa_append_kv: k_new, v_new, caches and positions are required");
    if (head_dim <= 0 || head_dim % 32)
        return fail(FA_ERR_HEAD_DIM, "fa_append_kv: head_dim %d must be a positive multiple of 32",
                    head_dim);
    if (n_kv_heads <= 0)
        return fail(FA_ERR_HEADS, "fa_append_kv: n_kv_heads %d", n_kv_heads);
    const bool paged = block_table != nullptr;
    if (batch < 0 || max_blocks_per_seq <= 0 ||
        (paged && (page_size <= 0 || page_size % 16 || num_blocks <= 0)))
        return fail(FA_ERR_LAYOUT, "fa_append_kv: bad batch, capacity, page size or block count");
    const long long cap = paged ? (long long)max_blocks_per_seq * page_size
                                : (long long)max_blocks_per_seq;
    const size_t new_bytes = (size_t)batch * n_kv_heads * head_dim * sizeof(float);
    const size_t rows = paged ? (size_t)num_blocks * page_size : (size_t)batch * cap;
    const size_t kv_rows = rows * n_kv_heads;
    const void *ins[3] = {k_new, v_new, positions};
    const size_t in_bytes[3] = {new_bytes, new_bytes, (size_t)batch * 4};
    for (int i = 0; i < 3; ++i)
        if (overlaps(k_cache, kv_rows * head_dim * 2, ins[i], in_bytes[i]) ||
            overlaps(v_cache, kv_rows * head_dim * (v_scales ? 1 : 2), ins[i], in_bytes[i]) ||
            (v_scales && overlaps(v_scales, kv_rows * (head_dim / 32) * 2, ins[i], in_bytes[i])))
            return fail(FA_ERR_ALIAS, "fa_append_kv: a cache overlaps k_new, v_new or positions");
    if (!aligned_to(k_new, 4) || !aligned_to(v_new, 4) || !aligned_to(positions, 4) ||
        !aligned_to(block_table, 4) || !aligned_to(k_cache, 2) ||
        !aligned_to(v_cache, v_scales ? 1 : 2) || !aligned_to(v_scales, 2))
        return fail(FA_ERR_ALIGN, "fa_append_kv: a pointer is not aligned to its element type");
    if ((long long)batch * n_kv_heads > 0x7fffffffll)
        return fail(FA_ERR_LAYOUT, "fa_append_kv: too many rows");
    if (batch == 0)
        return 0;
    Params p = {};
    memset(&p, 0, sizeof(p));
    p.bt = block_table;
    p.seq_lens = positions;
    p.B = batch;
    p.Hkv = n_kv_heads;
    p.page_size = paged ? page_size : 16;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.cap = cap;
    p.n_slots = batch;
    fa_append_kernel<<<batch * n_kv_heads, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        p, k_new, v_new, static_cast<__half *>(k_cache), v_cache,
        static_cast<__half *>(v_scales), head_dim);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(FA_ERR_CUDA, "fa_append_kv: launch failed: %s", cudaGetErrorString(e));
    return 0;
}

// Append into contiguous per-slot rings or rows: fa_append_kv_ring (one slot
// per sequence) and fa_append_kv_slots (slot map).
static int append_contig(const char *name, const float *k_new, const float *v_new, void *k_cache,
                         void *v_cache, void *v_scales, const int32_t *slot_ids,
                         const int32_t *positions, int batch, int n_kv_heads, int head_dim,
                         int n_slots, int capacity, bool ring, void *stream)
{
    g_err[0] = 0;
    if (!k_new || !v_new || !k_cache || !v_cache || !positions)
        return fail(FA_ERR_NULL, "%s: k_new, v_new, caches and positions are required", name);
    if (head_dim <= 0 || head_dim % 32)
        return fail(FA_ERR_HEAD_DIM, "%s: head_dim %d must be a positive multiple of 32", name,
                    head_dim);
    if (n_kv_heads <= 0)
        return fail(FA_ERR_HEADS, "%s: n_kv_heads %d", name, n_kv_heads);
    if (batch < 0 || capacity <= 0 || (ring && capacity % 16) || n_slots <= 0 ||
        (double)n_slots * n_kv_heads * (double)capacity > 1e15)
        return fail(FA_ERR_LAYOUT, "%s: bad batch, slot count or capacity (a multiple of 16 "
                                   "for a ring)", name);
    const size_t new_bytes = (size_t)batch * n_kv_heads * head_dim * sizeof(float);
    const size_t kv_rows = (size_t)n_slots * capacity * n_kv_heads;
    const void *ins[4] = {k_new, v_new, positions, slot_ids};
    const size_t in_bytes[4] = {new_bytes, new_bytes, (size_t)batch * 4, (size_t)batch * 4};
    for (int i = 0; i < 4; ++i)
        if (overlaps(k_cache, kv_rows * head_dim * 2, ins[i], in_bytes[i]) ||
            overlaps(v_cache, kv_rows * head_dim * (v_scales ? 1 : 2), ins[i], in_bytes[i]) ||
            (v_scales && overlaps(v_scales, kv_rows * (head_dim / 32) * 2, ins[i], in_bytes[i])))
            return fail(FA_ERR_ALIAS, "%s: a cache overlaps k_new, v_new, positions or slot_ids",
                        name);
    if (!aligned_to(k_new, 4) || !aligned_to(v_new, 4) || !aligned_to(positions, 4) ||
        !aligned_to(slot_ids, 4) || !aligned_to(k_cache, 2) ||
        !aligned_to(v_cache, v_scales ? 1 : 2) || !aligned_to(v_scales, 2))
        return fail(FA_ERR_ALIGN, "%s: a pointer is not aligned to its element type", name);
    if ((long long)batch * n_kv_heads > 0x7fffffffll)
        return fail(FA_ERR_LAYOUT, "%s: too many rows", name);
    if (batch == 0)
        return 0;
    Params p = {};
    memset(&p, 0, sizeof(p));
    p.seq_lens = positions;
    p.B = batch;
    p.Hkv = n_kv_heads;
    p.page_size = 16;
    p.max_blocks = capacity;
    p.cap = capacity;
    p.ring = ring ? 1 : 0;
    p.slot = slot_ids;
    p.n_slots = n_slots;
    fa_append_kernel<<<batch * n_kv_heads, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        p, k_new, v_new, static_cast<__half *>(k_cache), v_cache,
        static_cast<__half *>(v_scales), head_dim);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(FA_ERR_CUDA, "%s: launch failed: %s", name, cudaGetErrorString(e));
    return 0;
}

FA_API int fa_append_kv_ring(const float *k_new, const float *v_new, void *k_cache, void *v_cache,
                             void *v_scales, const int32_t *positions, int batch, int n_kv_heads,
                             int head_dim, int capacity, void *stream)
{
    return append_contig("fa_append_kv_ring", k_new, v_new, k_cache, v_cache, v_scales, nullptr,
                         positions, batch, n_kv_heads, head_dim, batch > 0 ? batch : 1, capacity,
                         true, stream);
}

FA_API int fa_append_kv_slots(const float *k_new, const float *v_new, void *k_cache,
                              void *v_cache, void *v_scales, const int32_t *slot_ids,
                              const int32_t *positions, int batch, int n_kv_heads, int head_dim,
                              int n_slots, int capacity, int ring, void *stream)
{
    if (!slot_ids) {
        g_err[0] = 0;
        return fail(FA_ERR_NULL, "fa_append_kv_slots: slot_ids is required");
    }
    return append_contig("fa_append_kv_slots", k_new, v_new, k_cache, v_cache, v_scales,
                         slot_ids, positions, batch, n_kv_heads, head_dim, n_slots, capacity,
                         ring != 0, stream);
}

FA_API int fa_gather_kv_debug(const void *cache, int row_bytes, const int32_t *block_table,
                              int b, int n_kv_heads, int page_size, int max_blocks_per_seq,
                              int num_blocks, int n_tokens, void *dense, void *stream)
{
    g_err[0] = 0;
    if (!cache || !dense)
        return fail(FA_ERR_NULL, "fa_gather_kv_debug: null pointer");
    const bool paged = block_table != nullptr;
    if (row_bytes <= 0 || n_kv_heads <= 0 || b < 0 || n_tokens < 0 || max_blocks_per_seq <= 0 ||
        (paged && (page_size <= 0 || page_size % 16 || num_blocks <= 0)))
        return fail(FA_ERR_LAYOUT, "fa_gather_kv_debug: bad sizes");
    const long long cap = paged ? (long long)max_blocks_per_seq * page_size : max_blocks_per_seq;
    if (n_tokens > cap)
        return fail(FA_ERR_LAYOUT, "fa_gather_kv_debug: n_tokens %d > capacity %lld", n_tokens,
                    cap);
    if (!aligned_to(block_table, 4))
        return fail(FA_ERR_ALIGN, "fa_gather_kv_debug: block_table must be 4-byte aligned");
    if (n_tokens == 0)
        return 0;
    Params p = {};
    memset(&p, 0, sizeof(p));
    p.k = static_cast<const char *>(cache);
    p.bt = block_table;
    p.Hkv = n_kv_heads;
    p.page_size = paged ? page_size : 16;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.cap = cap;
    fa_gather_kernel<<<dim3(n_tokens, n_kv_heads), 128, 0, static_cast<cudaStream_t>(stream)>>>(
        p, row_bytes, b, n_tokens, static_cast<unsigned char *>(dense));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(FA_ERR_CUDA, "fa_gather_kv_debug: launch failed: %s", cudaGetErrorString(e));
    return 0;
}

FA_API int fa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                             const void *v_scales, const int32_t *block_table,
                             const int32_t *seq_lens, int n_q_heads, int n_kv_heads,
                             int head_dim, float scale, const int32_t *window, void *out,
                             int batch, int page_size, int max_blocks_per_seq, int num_blocks,
                             void *stream)
{
    g_err[0] = 0;
    if (head_dim != 128 && head_dim != 256)
        return fail(FA_ERR_HEAD_DIM, "fa_decode_noalloc: head_dim %d not supported (128 or 256)",
                    head_dim);
    if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads)
        return fail(FA_ERR_HEADS, "fa_decode_noalloc: bad heads (q %d, kv %d)", n_q_heads,
                    n_kv_heads);
    if (batch < 0 || max_blocks_per_seq <= 0 || (block_table && page_size <= 0))
        return fail(FA_ERR_LAYOUT, "fa_decode_noalloc: bad batch, capacity or page size");
    const long long cap = block_table ? (long long)max_blocks_per_seq * page_size
                                      : (long long)max_blocks_per_seq;
    if (cap > (1ll << 30))
        return fail(FA_ERR_LAYOUT, "fa_decode_noalloc: capacity %lld tokens too large", cap);
    // the scratch this call needs: its own V type and the plan fa_decode takes
    const long long kv_rows_total =
        block_table ? (long long)(num_blocks > 0 ? num_blocks : 0) * n_kv_heads * page_size
                    : (long long)batch * n_kv_heads * cap;
    int sms = 0;
    Plan pl;
    size_t need = 0;
    const int prc = call_plan(batch, n_q_heads, n_kv_heads, head_dim, cap, v_scales != nullptr,
                              false, 1, 0, kv_rows_total, &sms, &pl, &need);
    if (prc)
        return prc;
    if (need > FA_NOALLOC_SCRATCH_BYTES)
        return fail(FA_ERR_WORKSPACE,
                    "fa_decode_noalloc: these sizes need %zu bytes of scratch, more than the "
                    "library's fixed %u bytes; use fa_decode with a caller workspace",
                    need, (unsigned)FA_NOALLOC_SCRATCH_BYTES);
    void *scratch = nullptr;
    const int rc = noalloc_scratch(&scratch);
    if (rc)
        return rc;
    return fa_decode(q, k_cache, v_cache, v_scales, block_table, seq_lens, n_q_heads,
                     n_kv_heads, head_dim, scale, window, out, batch, page_size,
                     max_blocks_per_seq, num_blocks, scratch, FA_NOALLOC_SCRATCH_BYTES, stream);
}

FA_API int fa_decode_profile_next(void *split_start, void *split_end)
{
    g_err[0] = 0;
    g_prof_start = static_cast<cudaEvent_t>(split_start);
    g_prof_end = static_cast<cudaEvent_t>(split_end);
    return 0;
}

FA_API int fa_selftest_wait_timeout(void *stream)
{
    g_err[0] = 0;
    fa_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(FA_ERR_CUDA, "fa_selftest_wait_timeout: launch failed: %s",
                    cudaGetErrorString(e));
    return 0;
}

FA_API int fa_decode_device_status(unsigned int *status, void *stream)
{
    g_err[0] = 0;
    if (!status)
        return fail(FA_ERR_NULL, "fa_decode_device_status: null pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int v = 0;
    const unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status, sizeof(v), 0,
                                              cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return fail(FA_ERR_CUDA, "fa_decode_device_status: %s", cudaGetErrorString(e));
    *status = v;
    return 0;
}

}  // extern "C"
