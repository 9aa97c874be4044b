// gemm_i4_tc.cu -- tensor-core (tcgen05, sm_103a) AutoRound int4 group-128 W4A8 GEMM.
//
// "radiance_autoround.py", module docstring and _exact_ref: symmetric int4 weights with one fp16
// scale per 128 input channels and output column, zero point 8 folded in, fp8 (e4m3) per-token
// activations, fp32 accumulation:
//   out[m,n] = bf16( x_scale[m] * sum_g s[g,n] * sum_{k in g} e4m3(xq[m,k]) * (c[k,n] - 8) ).
//
// The 4-bit code c itself, zero-extended to a byte, is the e4m3 encoding of c * 2^-9: codes 0-7
// are the subnormals m * 2^-9 and codes 8-15 the first normal binade (1 + m/8) * 2^-6, which
// continue the same linear scale.  So the operand tile is the codes spread to bytes (two masks
// and two byte permutes per eight codes), and the zero point rides on four more MMAs per k-tile
// whose A operand is the constant e4m3 -2^-6 (= -8 * 2^-9) in every element:
//   sum_k c_k 2^-9 x_k + sum_k (-8 * 2^-9) x_k = 2^-9 * sum_k (c_k - 8) x_k,
// all inputs exact, accumulated in fp32 tensor memory.  ((c - 8) * 2^-9 is an exact e4m3 value
// too, and the prefill kernel (gemm_i4_pf.cu) builds it with three byte permutes per four codes;
// at decode even that makes the converter warps the busiest unit, 48 -> 52 us for gate_up at M=1,
// so this kernel keeps the nibble bytes and the four extra MMAs.)  With
// per-column zero points (asymmetric) the constant-operand MMAs write a second accumulator,
// which the promotion scales by z / 8.  The group scale is not a power of two and cannot ride on
// the instruction's block scale, so each group's partial is read back and promoted into fp32
// registers as acc += (512 * s[g,n]) * partial.
//
//   * swap-AB as in the MXFP4 kernel: the weights are the MMA "M" operand (128 output columns n
//     per tile, one per tensor-memory lane) and the tokens the "N" operand (16, 32 or 64);
//   * TMA brings the checkpoint words as stored ([K/8, N] int32, 8 consecutive k of one column
//     per word, 512 contiguous bytes per box row) plus the activation tiles;
//   * eight converter warps turn each k-tile (128 k x 128 columns) into the e4m3 operand tile the
//     instruction reads (K-major, 128-byte swizzle); the constant zero-point operand is one 1 KB
//     swizzle atom that every 8-row group of the instruction reads (stride 0);
//   * a k-tile is one group, so every k-tile's MMAs go to a fresh accumulator buffer in
//     tensor memory (four buffers rotate); four promotion warps read it, scale by s[g,n] (read
//     from global memory a unit ahead) and add into registers; at the end of a tile the same
//     warps write bf16 through a shared-memory stage and TMA stores, or the fp32 partial of a
//     split tile for the stream-K fix-up (last contributor adds partials in CTA order);
//   * the work split, bounded waits, gate warp and abort handling follow the MXFP4 kernel.
//
// int5 ("vllm-radiance (MXFP4)", section "int5 (W5A8)": 5-bit codes c, value c - 16, the low
// nibbles in the same word layout and the fifth bit in a plane of one byte per word, bit j of
// byte (i, n) for k = 8i + j).  (c - 16) * 2^-9 is exact in e4m3 as well: for c >= 16 it is the
// nibble's own byte (0x00-0x0F), for c < 16 the sign bit over 16 - nibble, i.e. 0x90 - nibble
// (0x10 is 2^-5 = 16 * 2^-9).  So the fifth bit only picks between the nibble and 0x90 - nibble,
// and the symmetric int5 kernel needs no zero-point MMAs at all (here the converter's extra work
// pays: a separate fifth-bit operand tile would cost its stores and four MMAs).  With a zero
// point z per (group, column) the constant-atom MMAs write the group sums into the second
// accumulator as for asymmetric int4, and promotion adds ((z - 16) / 8) times it.
//
// Warp roles: 0 TMA producer, 1 TMEM allocator + MMA issuer, 5 gate, 2-4, 6-8, 10, 11 converters,
// 12-15 promotion and epilogue (9 idle).
#include <algorithm>
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "dispatch.h"
#include "tc_host.cuh"
#include "tc_ptx.cuh"
#include "tc_sched.cuh"
#include "wcodes.cuh"

namespace w4a8 {
namespace tci {

using namespace tcs;

// Warp w issues from scheduler w % 4.  The scheduler of the MMA-issuing warp loses issue cycles
// while MMAs go out, so it hosts only the MMA warp, the gate and the one promotion warp that its
// tensor-memory lane quarter forces there; the eight converter warps sit on the other three.
constexpr int NUM_THREADS = 512;  // 16 warps
constexpr int MMA_WARP = 1;
constexpr int GATE_WARP = 5;      // warp 9 has no role
constexpr int EPI_WARP0 = 12;     // warps 12-15: promotion + epilogue, lane quarter = warp & 3
constexpr int N_CONV_WARPS = 8;   // warps 2, 3, 4, 6, 7, 8, 10, 11
// 64-token tiles without zero points: the promotion warps (warpgroup 3) hold 64 accumulators
// plus a 16-column load; at the launch's 128 registers per thread that spilled, and with shared
// memory filling the L1 array every reload is an L2 round trip.  So those builds move registers
// from warpgroups 0-2 to warpgroup 3 with setmaxnreg (the asymmetric builds spill more under
// any split, so they keep 128 everywhere).
constexpr int REGS_REST_BN64 = 112;
constexpr int REGS_EPI_BN64 = 136;
static_assert(3 * 128 * REGS_REST_BN64 + 128 * REGS_EPI_BN64 <= NUM_THREADS * 118, "register split");

// Converter index 0..7 of a warp, or -1.
__device__ __forceinline__ int conv_index(int warp)
{
    switch (warp) {
    case 2: return 0;
    case 3: return 1;
    case 4: return 2;
    case 6: return 3;
    case 7: return 4;
    case 8: return 5;
    case 10: return 6;
    case 11: return 7;
    default: return -1;
    }
}
constexpr int GATE_BARRIER = 2;
constexpr int KPU = 4;            // k-tiles per ring fill: one 4-k-tile unit

enum : unsigned { ST_TIMEOUT_PRODUCER = 1, ST_TIMEOUT_GATE = 2, ST_TIMEOUT_CONV = 4, ST_TIMEOUT_EPI = 8 };

struct Params {
    const uint16_t *s16;   // [K/128, N] fp16 group scales
    const float *xs;       // [M] per-token scale
    const int32_t *qz;     // asymmetric int4 only: [K/128, ceil(N/8)] packed zero points minus one
    const uint8_t *z5;     // asymmetric int5 only: [K/128, N] zero points
    uint16_t *out;         // [M, N] bf16
    float *partials;       // [G][2][BN][128] fp32 stream-K partial tiles
    int *counters;         // arrival counters of the split tiles (index < G), zero between calls
    unsigned int *status;  // device status block
    int M, N, K;
    int m_tiles, n_tiles;
    int U;                 // 4-k-tile units per tile
    long long RU;          // stream-K units
    int R, D, G, Gsk;      // work split (see Sched)
    int tma_out;           // output through TMA stores (else plain stores)
    unsigned long long *trace;  // optional pipeline timeline of CTA 0 (diagnostics), or null
};

// Pipeline timeline (a development aid, compiled in only when W4A8_TRACE is defined): CTA 0
// records clock64() per k-tile i < 256 for each event:
// 0 fill issued (index = fill), 1 converter start, 2 converter done, 3 MMA released,
// 4 promotion start, 5 promotion done, 6 MMA warp met the gate, 7-14 each converter warp done.
__device__ __forceinline__ void trace_ev(const Params &p, int ev, int i)
{
#ifdef W4A8_TRACE
    if (p.trace != nullptr && blockIdx.x == 0 && i < 256) p.trace[ev * 256 + i] = (unsigned long long)clock64();
#endif
}

// Shared memory: the zero-point operand atom (1 KB), NA converted operand tiles, then a ring of
// US fills, each holding KPU k-tiles of activations
// (BN x 128 bytes, swizzled) and of checkpoint words ([16 word rows][128 columns]), then (int5)
// KPU k-tiles of the fifth-bit plane ([16 byte rows][128 columns]).
template <int BN, int US, int NA, int NB, bool ASYM = false, bool I5 = false>
struct Layout {
    static constexpr int RAW_TILE = 16 * BM * 4;  // 8 KB of words: 128 k x 128 columns
    static constexpr int PLANE_TILE = I5 ? 16 * BM : 0;  // 2 KB of fifth bits: 128 k x 128 columns
    static constexpr int X_TILE = BN * 128;
    static constexpr int A_TILE = BM * 128;       // e4m3 [128 columns][128 k], 128-byte swizzle
    static constexpr int RAW_SLOT = KPU * (RAW_TILE + PLANE_TILE);
    static constexpr int PLANE_OFF = KPU * RAW_TILE;  // within a raw slot
    static constexpr int X_SLOT = KPU * X_TILE;
    static constexpr int Z_OFF = 0;                // 8 rows x 128 bytes of e4m3 -2^-6
    static constexpr int A_OFF = Z_OFF + 1024;
    static constexpr int X_OFF = A_OFF + NA * A_TILE;
    static constexpr int RAW_OFF = X_OFF + US * X_SLOT;
    static constexpr int BAR_OFF = RAW_OFF + US * RAW_SLOT;
    static constexpr int XS_OFF = BAR_OFF + 512;
    static constexpr int NSTAGE = BN == 16 ? 1 : 2;
    static constexpr int STAGE_BYTES = 16 * BM * 2;
    static constexpr int STAGE_OFF = (XS_OFF + BN * 4 + 1023) / 1024 * 1024;
    static constexpr int TOTAL = STAGE_OFF + NSTAGE * STAGE_BYTES + 1024;  // + alignment slack
    static constexpr int TX_BYTES = KPU * (RAW_TILE + PLANE_TILE + X_TILE);
    static constexpr int TMEM_NEED = NB * BN * (ASYM ? 2 : 1);  // + the zero-point sums (asymmetric)
    static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128
                                     : TMEM_NEED <= 256 ? 256 : 512;
    static_assert(TMEM_NEED <= 512, "tensor memory");
    static_assert(TOTAL <= 232448, "shared memory");
    static_assert((X_TILE % 1024) == 0 && (X_OFF % 1024) == 0 && (A_TILE % 1024) == 0, "swizzled tiles");
    static_assert(8 * (2 * US + NA + 2 * NB + 1) + 32 <= 512, "barrier area");
    static_assert(NA <= NB, "a converted tile's release rides on the group-accumulator barrier");
};

template <int BN, int US, int NA, int NB, bool ASYM, bool I5>
__global__ void __launch_bounds__(NUM_THREADS, 1)
int4_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_x,
               const __grid_constant__ CUtensorMap tmap_out, const __grid_constant__ CUtensorMap tmap_h,
               const Params p)
{
    using L = Layout<BN, US, NA, NB, ASYM, I5>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);  // ring fill landed
    uint64_t *empty = full + US;                                        // ring fill consumed by the MMAs
    uint64_t *a_full = empty + US;                                      // converted tile written
    uint64_t *g_full = a_full + NA;  // a k-tile's MMAs done: its group accumulator is complete and
                                     // its converted tile free again (one commit serves both)
    uint64_t *g_empty = g_full + NB;                                    // group accumulator promoted
    uint64_t *mma_done = g_empty + NB;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *last_flag = reinterpret_cast<int *>(tmem_slot + 2);
    int *issued = reinterpret_cast<int *>(tmem_slot + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const Sched sched(cta, p.Gsk, p.RU, p.D, p.R, p.U);
    const int n_k = 4 * sched.n_units;  // k-tiles (= groups) this CTA processes

    if (threadIdx.x == 0) {
        for (int s = 0; s < US; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < NA; ++a) tc::mbar_init(&a_full[a], N_CONV_WARPS);  // one arrival per converter warp
        for (int b = 0; b < NB; ++b) {
            tc::mbar_init(&g_full[b], 1);
            tc::mbar_init(&g_empty[b], 4);  // one arrival per promotion warp
        }
        tc::mbar_init(mma_done, 1);
        *abort_flag = 0;
        *last_flag = 0;
        *issued = 0;
        tc::fence_mbar_init();
        tc::tma_prefetch_desc(&tmap_q);
        tc::tma_prefetch_desc(&tmap_x);
        if (I5) tc::tma_prefetch_desc(&tmap_h);
        if (p.tma_out) tc::tma_prefetch_desc(&tmap_out);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, L::TMEM_COLS);
        tc::tmem_relinquish();
    }
    // the zero-point operand atom (a swizzle only permutes its equal bytes), made visible to the
    // tensor core before the barrier below; the symmetric int5 kernel does not read it
    if ((!I5 || ASYM) && threadIdx.x < 64) {
        const uint32_t z = E4M3_MINUS_2POW_M6 * 0x01010101u;
        reinterpret_cast<uint4 *>(smem + L::Z_OFF)[threadIdx.x] = make_uint4(z, z, z, z);
        tc::fence_proxy_async_smem();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // programmatic dependent launch: global memory only after the previous kernel completed
    tc::grid_dependency_wait();
    tc::grid_dependents_launch();
    if constexpr (BN >= 64 && !ASYM) {
        if (warp >= EPI_WARP0)
            tc::regs_inc<REGS_EPI_BN64>();
        else
            tc::regs_dec<REGS_REST_BN64>();
    }

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int i = 0; i < n_k && !*abort_flag; i += KPU) {
                int kt, n0;
                sched.fill_at(i, p.m_tiles, kt, n0);
                const long long u = sched.unit_at(i / 4);
                const int m0 = ((int)div_nonneg(u, p.U) % p.m_tiles) * BN;
                const int f = i / KPU, sl = f % US;
                if (wait_or_fail(&empty[sl], ((f / US) & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER, f))
                    break;
                tc::mbar_arrive_expect_tx(&full[sl], L::TX_BYTES);
                tc::tma_load_2d(smem + L::RAW_OFF + sl * L::RAW_SLOT, &tmap_q, &full[sl], n0, 16 * kt);
                tc::tma_load_3d(smem + L::X_OFF + sl * L::X_SLOT, &tmap_x, &full[sl], 0, m0, kt);
                if constexpr (I5)
                    tc::tma_load_2d(smem + L::RAW_OFF + sl * L::RAW_SLOT + L::PLANE_OFF, &tmap_h, &full[sl], n0, 16 * kt);
                *issued = f + 1;
                trace_ev(p, 0, f);
            }
        }
        __syncwarp();
    } else if (conv_index(warp) >= 0) {
        // ------------------------------------------------------------ converters (2-5, 11-14)
        // Thread = one weight column of the tile (row of the MMA operand) and one half of the
        // k-tile: it reads its 8 words (conflict-free: consecutive columns are consecutive words),
        // writes the 64 e4m3 codes as four 16-byte chunks at their swizzled places, and the eight
        // warps publish the tile together.
        const int ci = conv_index(warp);
        const int r = 32 * (ci >> 1) + lane;
        const int h = ci & 1;
        int w = 0;
        for (int i = 0; i < n_k; ++i) {
            const int f = i / KPU, sl = f % US, j = i % KPU, a = i % NA;
            if (j == 0 && (w = warp_wait(&full[sl], (f / US) & 1, abort_flag, p.status, ST_TIMEOUT_CONV, f, lane)))
                break;
            // the tile slot is free once the MMAs of k-tile i - NA are done: that k-tile's g_full
            // phase (it cannot be a phase behind, as k-tile i + 1 - NA + NB needs this tile first)
            if (i >= NA && (w = warp_wait(&g_full[(i - NA) % NB], ((i - NA) / NB) & 1, abort_flag, p.status,
                                          ST_TIMEOUT_CONV, i, lane)))
                break;
            if (ci == 0 && lane == 0) trace_ev(p, 1, i);
            const uint32_t *raw = reinterpret_cast<const uint32_t *>(smem + L::RAW_OFF + sl * L::RAW_SLOT) + j * 16 * BM + r;
            uint8_t *dst = smem + L::A_OFF + a * L::A_TILE + r * 128;
            uint32_t wv[8];  // all 8 words first, so the conversions below run side by side
#pragma unroll
            for (int k = 0; k < 8; ++k) wv[k] = raw[(8 * h + k) * BM];
            uint32_t hb[8];  // int5: the plane bytes of the same word rows (one per word)
            if constexpr (I5) {
                const uint8_t *pl = smem + L::RAW_OFF + sl * L::RAW_SLOT + L::PLANE_OFF + (j * 16 + 8 * h) * BM + r;
#pragma unroll
                for (int k = 0; k < 8; ++k) hb[k] = pl[k * BM];
            }
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {  // 16-byte chunk c = k 16c .. 16c+15 = words 2c, 2c+1
                const int c = 4 * h + cc;
                uint2 lo, hi;
                if constexpr (I5) {
                    lo = i5x8_to_signed_bytes(wv[2 * cc], hb[2 * cc]);
                    hi = i5x8_to_signed_bytes(wv[2 * cc + 1], hb[2 * cc + 1]);
                } else {
                    lo = i4x8_to_bytes(wv[2 * cc]);
                    hi = i4x8_to_bytes(wv[2 * cc + 1]);
                }
                *reinterpret_cast<uint4 *>(dst + ((c ^ (r & 7)) << 4)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
            }
            tc::fence_proxy_async_smem();  // generic writes -> visible to the tensor core
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&a_full[a]);
            if (ci == 0 && lane == 0) trace_ev(p, 2, i);
            if (lane == 0) trace_ev(p, 7 + ci, i);
        }
    } else if (warp == MMA_WARP || warp == GATE_WARP) {
        // ------------------------------------------------------------ MMA issuer and its gate
        // As in the MXFP4 kernel: the gate does the mbarrier waiting (group buffer free, converted
        // tile ready) and releases the MMA warp through a named barrier once per k-tile.
        const bool gate = (warp == GATE_WARP);
        if (!gate) tc::tc_fence_after();
        const uint32_t idesc = tc::idesc_f8f6f4(0, 0, BM, BN);
        for (int i = 0; i < n_k; ++i) {
            const int f = i / KPU, sl = f % US, j = i % KPU, a = i % NA, b = i % NB;
            if (gate && lane == 0) {  // lane 0 waits, the converted tile first; the barrier releases the rest
                if (!*abort_flag) wait_or_fail(&a_full[a], (i / NA) & 1, abort_flag, p.status, ST_TIMEOUT_GATE, i);
                if (!*abort_flag)
                    wait_or_fail(&g_empty[b], ((i / NB) & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_GATE, i);
                trace_ev(p, 3, i);
            }
            const bool aborted = tc::named_bar_or(GATE_BARRIER, 64, gate && *abort_flag);
            if (gate && lane == 0) trace_ev(p, 6, i);
            if (!gate && lane == 0 && !aborted) {
                tc::tc_fence_after();
                const uint32_t aa = tc::smem_u32(smem + L::A_OFF + a * L::A_TILE);
                const uint32_t za = tc::smem_u32(smem + L::Z_OFF);
                const uint32_t xa = tc::smem_u32(smem + L::X_OFF + sl * L::X_SLOT + j * L::X_TILE);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_f8f6f4(tmem + b * BN, tc::smem_desc(aa + 32 * kk, 16, 1024, 2),
                                   tc::smem_desc(xa + 32 * kk, 16, 1024, 2), idesc, kk > 0 ? 1u : 0u);
                // zero point: the constant atom for every 8-row group (stride 0), into the same
                // accumulator (int4, zero point 8), or with per-column zero points into a buffer of
                // its own, scaled per column in promotion; the symmetric int5 operand holds c - 16
                if constexpr (!I5 || ASYM) {
                    const uint32_t zacc = tmem + (ASYM ? NB + b : b) * BN;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_f8f6f4(zacc, tc::smem_desc(za + 32 * kk, 16, 0, 2),
                                       tc::smem_desc(xa + 32 * kk, 16, 1024, 2), idesc, (ASYM && kk == 0) ? 0u : 1u);
                }
                tc::tc_commit(&g_full[b]);
                if (j == KPU - 1) tc::tc_commit(&empty[sl]);
            }
            __syncwarp();
        }
        if (!gate && lane == 0) tc::tc_commit(mma_done);  // teardown waits on it before freeing TMEM
        __syncwarp();
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------------------ promotion and epilogue (12-15)
        const int q = warp & 3;
        const int r = 32 * q + lane;  // weight column of the tile = TMEM lane
        const bool issuer = (threadIdx.x == EPI_WARP0 * 32);
        int ck = 0;  // output chunks emitted (staging buffer rotation)
        // 16 token columns of this thread's weight column: through a [16 tokens][128 columns] bf16
        // stage and one TMA store (all 128 threads call together), or plain stores.
        auto emit = [&](const float (&o)[16], int c0, int m0, int n0) {
            const int n = n0 + r;
            if (p.tma_out) {
                uint16_t *stg = reinterpret_cast<uint16_t *>(smem + L::STAGE_OFF + (ck % L::NSTAGE) * L::STAGE_BYTES);
                if (ck >= L::NSTAGE) {
                    if (issuer) tc::bulk_wait_group_read<L::NSTAGE - 1>();
                    tc::named_bar_sync(1, 128);
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) stg[j * BM + r] = float_to_bf16_bits(o[j]);
                tc::fence_proxy_async_smem();
                tc::named_bar_sync(1, 128);
                if (issuer) {
                    tc::tma_store_2d(&tmap_out, stg, n0, m0 + c0);
                    tc::bulk_commit_group();
                }
                ++ck;
            } else if (n < p.N) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (m0 + c0 + j < p.M) tc::st_cg_u16(p.out + (size_t)(m0 + c0 + j) * p.N + n, float_to_bf16_bits(o[j]));
            }
        };
        // group scales of one unit (4 k-tiles) for this thread's column, times 2^9 (the operand
        // codes are c * 2^-9), fetched a unit ahead
        auto unit_scales = [&](int pu, float (&dst)[4]) {
            if (pu >= sched.n_units) return;
            const long long u = sched.unit_at(pu);
            const int t = (int)div_nonneg(u, p.U);
            const int n = (t / p.m_tiles) * BM + r;
            const int g0 = (int)(u - (long long)t * p.U) * 4;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                dst[jj] = n < p.N ? 512.0f * __half2float(__ushort_as_half(__ldg(p.s16 + (size_t)(g0 + jj) * p.N + n))) : 0.0f;
        };
        // asymmetric: the unit's zero points z of this thread's column, as z / 8 for int4 (the
        // accumulator holds the codes alone) or (z - 16) / 8 for int5 (it holds c - 16); exact
        auto unit_zeros = [&](int pu, float (&dst)[4]) {
            if (pu >= sched.n_units) return;
            const long long u = sched.unit_at(pu);
            const int t = (int)div_nonneg(u, p.U);
            const int n = (t / p.m_tiles) * BM + r;
            const int g0 = (int)(u - (long long)t * p.U) * 4;
            const int nz = (p.N + 7) / 8;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                if constexpr (I5) {
                    const int z = n < p.N ? (int)__ldg(p.z5 + (size_t)(g0 + jj) * p.N + n) : 16;
                    dst[jj] = 0.125f * (float)(z - 16);
                } else {
                    const uint32_t w = n < p.N ? (uint32_t)__ldg(p.qz + (size_t)(g0 + jj) * nz + n / 8) : 0x77777777u;
                    dst[jj] = 0.125f * (float)(1 + ((w >> (4 * (n & 7))) & 0xfu));
                }
            }
        };
        float sc_cur[4] = {0.0f, 0.0f, 0.0f, 0.0f}, sc_nxt[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float zf_cur[4] = {1.0f, 1.0f, 1.0f, 1.0f}, zf_nxt[4] = {1.0f, 1.0f, 1.0f, 1.0f};
        unit_scales(0, sc_nxt);
        if (ASYM) unit_zeros(0, zf_nxt);
        int i = 0;  // k-tile position, in the order the MMAs run
        for (int seg = 0; seg < sched.S; ++seg) {
            long long u, ue;
            sched.seg_units(seg, u, ue);
            const int t = (int)div_nonneg(u, p.U);
            const long long t_lo = (long long)t * p.U, t_hi = t_lo + p.U;
            const bool whole = (u == t_lo) && (ue == t_hi);
            const int n0 = (t / p.m_tiles) * BM, m0 = (t % p.m_tiles) * BN;
            float *xs_s = reinterpret_cast<float *>(smem + L::XS_OFF);
            for (int c = r; c < BN; c += BM) xs_s[c] = (m0 + c < p.M) ? __ldg(p.xs + m0 + c) : 0.0f;
            float acc[BN];
#pragma unroll
            for (int c = 0; c < BN; ++c) acc[c] = 0.0f;
            bool gave_up = false;
            for (const int i_end = i + 4 * (int)(ue - u); i < i_end; ++i) {
                const int b = i % NB, jj = i & 3;
                if (jj == 0) {
#pragma unroll
                    for (int z = 0; z < 4; ++z) sc_cur[z] = sc_nxt[z];
                    unit_scales(i / 4 + 1, sc_nxt);
                    if (ASYM) {
#pragma unroll
                        for (int z = 0; z < 4; ++z) zf_cur[z] = zf_nxt[z];
                        unit_zeros(i / 4 + 1, zf_nxt);
                    }
                }
                int w = 0;
                if (lane == 0) w = tc::mbar_wait(&g_full[b], (i / NB) & 1, abort_flag, WAIT_BUDGET);
                w = __shfl_sync(0xffffffffu, w, 0);
                if (w) {
                    if (lane == 0) {
                        if (w == 1) fail(p.status, ST_TIMEOUT_EPI, &g_full[b], i);
                        *abort_flag = 1;
                    }
                    gave_up = true;
                    break;
                }
                tc::tc_fence_after();
                if (issuer) trace_ev(p, 4, i);
                const float s = jj == 0 ? sc_cur[0] : jj == 1 ? sc_cur[1] : jj == 2 ? sc_cur[2] : sc_cur[3];
                const uint32_t tb = tmem + b * BN + ((32u * q) << 16);
#pragma unroll
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    uint32_t v[16];
                    tc::tmem_ld16(tb + c0, v);
                    tc::tmem_ld_wait();
                    if constexpr (ASYM) {
                        // 512 s (P + (z/8) Z) = s (sum c x - z sum x), Z = -2^-6 sum x (int4); for
                        // int5 P holds c - 16 and the factor is (z - 16) / 8
                        const float zf = jj == 0 ? zf_cur[0] : jj == 1 ? zf_cur[1] : jj == 2 ? zf_cur[2] : zf_cur[3];
                        uint32_t vz[16];
                        tc::tmem_ld16(tb + NB * BN + c0, vz);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            acc[c0 + j] = fmaf(s, fmaf(zf, __uint_as_float(vz[j]), __uint_as_float(v[j])), acc[c0 + j]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[c0 + j] = fmaf(s, __uint_as_float(v[j]), acc[c0 + j]);
                    }
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&g_empty[b]);
                if (issuer) trace_ev(p, 5, i);
            }
            // all four warps leave together if any gave up (this also publishes xs_s)
            if (tc::named_bar_or(1, 128, gave_up)) break;
            if (whole) {
#pragma unroll
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    if (m0 + c0 < p.M) {
                        float o[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) o[j] = acc[c0 + j] * xs_s[c0 + j];
                        emit(o, c0, m0, n0);
                    }
                }
            } else {
                // stream-K: store this CTA's fp32 partial; the last contributor adds all in CTA order
                float *slot = p.partials + ((size_t)cta * 2 + (t == sched.t_first ? 0 : 1)) * (size_t)(BM * BN);
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (m0 + c < p.M) tc::st_cg_f32(slot + c * BM + r, acc[c]);  // tokens that exist
                const int c_first = unit_owner(t_lo, p.RU, p.Gsk);
                const int c_last = unit_owner(t_hi - 1, p.RU, p.Gsk);
                tc::named_bar_sync(1, 128);
                if (issuer) {
                    const int old = tc::atomic_add_acq_rel_gpu(p.counters + t, 1);
                    *last_flag = (old == c_last - c_first);
                }
                tc::named_bar_sync(1, 128);
                if (*last_flag) {
                    const int m_cnt = min(BN, p.M - m0);
                    for (int c0 = 0; c0 < m_cnt; c0 += 16) {
                        float sum[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) sum[j] = 0.0f;
                        for (int cb = c_first; cb <= c_last; cb += 4) {
                            float v[4][16];
#pragma unroll
                            for (int cc = 0; cc < 4; ++cc) {
                                const int c = min(cb + cc, c_last);  // past the end: reload the last, unused
                                const int sl = (t == (int)(unit_start(c, p.RU, p.Gsk) / p.U)) ? 0 : 1;
                                const float *src = p.partials + ((size_t)c * 2 + sl) * (size_t)(BM * BN) + c0 * BM + r;
#pragma unroll
                                for (int j = 0; j < 16; ++j) v[cc][j] = c0 + j < m_cnt ? __ldcg(src + j * BM) : 0.0f;
                            }
#pragma unroll
                            for (int cc = 0; cc < 4; ++cc)
                                if (cb + cc <= c_last) {
#pragma unroll
                                    for (int j = 0; j < 16; ++j) sum[j] += v[cc][j];
                                }
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) sum[j] *= xs_s[c0 + j];
                        emit(sum, c0, m0, n0);
                    }
                    if (issuer) p.counters[t] = 0;
                }
                tc::named_bar_sync(1, 128);  // last_flag is reused by the next tile
            }
        }
        if (issuer) tc::bulk_wait_group_all();  // output stores done before shared memory goes away
    }

    tc::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        int zero = 0;
        if (*abort_flag)  // drain: TMA copies issued but not waited for
            for (int f = max(0, *issued - US); f < *issued; ++f)
                if (tc::mbar_wait(&full[f % US], (f / US) & 1, &zero, DRAIN_BUDGET)) break;
        tc::mbar_wait(mma_done, 0, &zero, WAIT_BUDGET);  // every MMA finished before TMEM is freed
    }
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// ------------------------------------------------------------------------------- host side

struct Cfg {
    int BN, m_tiles, n_tiles, U;
    SkSplit k;
};

static Cfg choose(int64_t M, int64_t N, int64_t K)
{
    Cfg c;
    c.BN = M <= 16 ? 16 : M <= 32 ? 32 : 64;
    c.n_tiles = (int)((N + BM - 1) / BM);
    c.m_tiles = (int)((M + c.BN - 1) / c.BN);
    c.U = (int)(K / 512);
    c.k = sk_split((long long)c.n_tiles * c.m_tiles, c.U, tch::num_sms());
    return c;
}

static size_t partial_bytes(const Cfg &c)
{
    const size_t b = (size_t)c.k.G * 2 * BM * c.BN * 4;
    return (b + 255) / 256 * 256;
}

template <int BN, int US, int NA, int NB, bool ASYM, bool I5 = false>
static w4a8_status launch(const int32_t *qw, const uint8_t *xq, Params prm, cudaStream_t stream,
                          const uint8_t *qh = nullptr)
{
    using L = Layout<BN, US, NA, NB, ASYM, I5>;
    CUtensorMap tq, tx, tout, th;
    memset(&tout, 0, sizeof(tout));
    memset(&th, 0, sizeof(th));
    // int5 fifth-bit plane [K/8 rows][N columns] uint8: boxes of 16 * KPU byte rows x 128 columns
    if (I5 && !tch::tmap_2d(&th, CU_TENSOR_MAP_DATA_TYPE_UINT8, qh, prm.K / 8, prm.N, (uint64_t)prm.N, 16 * KPU,
                            BM, CU_TENSOR_MAP_SWIZZLE_NONE))
        return W4A8_ERR_CUDA;
    prm.tma_out = (prm.N % 8 == 0) && w4a8_aligned(prm.out, 16) &&
                  tch::tmap_2d(&tout, CU_TENSOR_MAP_DATA_TYPE_UINT16, prm.out, prm.M, prm.N, (uint64_t)prm.N * 2, 16,
                               BM, CU_TENSOR_MAP_SWIZZLE_NONE);
    // checkpoint words [K/8 rows][N columns] int32: a box is 16 * KPU word rows x 128 columns;
    // activations as in the MXFP4 kernel: [k-tile][row][128 bytes], 128-byte swizzle
    if (!tch::tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_INT32, qw, prm.K / 8, prm.N, (uint64_t)prm.N * 4, 16 * KPU, BM,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !tch::tmap_3d_ktiles(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, prm.M, prm.K, 128, prm.K / 128, BN, KPU))
        return W4A8_ERR_CUDA;
    auto kern = int4_tc_kernel<BN, US, NA, NB, ASYM, I5>;
    if constexpr (BN >= 64 && !ASYM) {
        // the register split assumes at least 118 registers per thread at launch; a build with
        // fewer would leave setmaxnreg.inc waiting, so it is refused
        static std::atomic<int> regs_state{0};  // 0 unknown, 1 enough, 2 too few
        int rs = regs_state.load(std::memory_order_acquire);
        if (rs == 0) {
            cudaFuncAttributes fa;
            rs = (cudaFuncGetAttributes(&fa, kern) == cudaSuccess && fa.numRegs >= 118) ? 1 : 2;
            regs_state.store(rs, std::memory_order_release);
        }
        if (rs != 1) return W4A8_ERR_CUDA;
    }
    static std::atomic<int> attr_done[64];
    if (!tch::set_smem_once(kern, L::TOTAL, attr_done)) return W4A8_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(prm.G);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = L::TOTAL;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tq, tx, tout, th, prm) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return w4a8_launch_status();
}

}  // namespace tci
}  // namespace w4a8

using namespace w4a8::tci;

bool w4a8_tc_int4_supported(const void *xq, const void *qw, const void *s16, const void *out, int64_t M,
                            int64_t N, int64_t K)
{
    // TMA: 16-byte aligned word rows (N a multiple of 4), whole 4-k-tile units (K % 512)
    if (K % 512 != 0 || K > (1ll << 30) || M < 1 || M > (1ll << 30) || N < 4 || N % 4 != 0 || N > (1ll << 30))
        return false;
    if (!w4a8_aligned(qw, 16) || !w4a8_aligned(xq, 16) || !w4a8_aligned(s16, 2) || !w4a8_aligned(out, 2))
        return false;
    return w4a8::tch::encode_fn() != nullptr;
}

size_t w4a8_tc_int4_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (K % 512 != 0 || K <= 0 || M <= 0 || N <= 0) return 0;
    const Cfg c = w4a8::tci::choose(M, N, K);
    const size_t own = W4A8_COUNTER_BYTES + partial_bytes(c);
    // prefill sizes may take the 256-token kernel instead: enough for either
    return M > W4A8_INT4_PF_MIN_M ? std::max(own, w4a8_int4_pf_workspace_bytes(M, N, K)) : own;
}

static bool make_params(Params &prm, const Cfg &c, const float *x_scale, const uint16_t *s16, uint16_t *out,
                        int64_t M, int64_t N, int64_t K, void *workspace)
{
    prm.s16 = s16;
    prm.xs = x_scale;
    prm.qz = nullptr;
    prm.z5 = nullptr;
    prm.out = out;
    if (c.k.G > W4A8_MAX_COUNTERS) return false;  // split tiles are indexed below the grid size
    prm.counters = static_cast<int *>(workspace);
    prm.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + W4A8_COUNTER_BYTES);
    prm.status = w4a8_device_status_ptr();
    prm.M = (int)M;
    prm.N = (int)N;
    prm.K = (int)K;
    prm.m_tiles = c.m_tiles;
    prm.n_tiles = c.n_tiles;
    prm.U = c.U;
    prm.RU = c.k.RU;
    prm.R = c.k.R;
    prm.D = c.k.D;
    prm.G = c.k.G;
    prm.Gsk = c.k.Gsk;
    prm.tma_out = 0;
    prm.trace = static_cast<unsigned long long *>(w4a8_debug_trace_ptr());
    return prm.status != nullptr;
}

w4a8_status w4a8_launch_int4_tc(const uint8_t *xq, const float *x_scale, const int32_t *qw, const uint16_t *s16,
                                uint16_t *out, int64_t M, int64_t N, int64_t K, void *workspace, int,
                                cudaStream_t stream, const int32_t *qzeros)
{
    if (qzeros == nullptr && w4a8_int4_pf_takes(M, false))
        return w4a8_launch_int4_pf(xq, x_scale, qw, nullptr, s16, out, M, N, K, workspace, stream);
    const Cfg c = w4a8::tci::choose(M, N, K);
    Params prm;
    if (!make_params(prm, c, x_scale, s16, out, M, N, K, workspace)) return W4A8_ERR_CUDA;
    prm.qz = qzeros;
    if (qzeros != nullptr) {
        switch (c.BN) {
        case 16: return launch<16, 4, 3, 4, true>(qw, xq, prm, stream);
        case 32: return launch<32, 3, 3, 4, true>(qw, xq, prm, stream);
        default: return launch<64, 2, 3, 4, true>(qw, xq, prm, stream);
        }
    }
    switch (c.BN) {
    case 16: return launch<16, 4, 3, 4, false>(qw, xq, prm, stream);
    case 32: return launch<32, 3, 3, 4, false>(qw, xq, prm, stream);
    default: return launch<64, 2, 3, 4, false>(qw, xq, prm, stream);
    }
}

bool w4a8_tc_int5_supported(const void *xq, const void *qw, const void *qh, const void *s16, const void *out,
                            int64_t M, int64_t N, int64_t K)
{
    // the fifth-bit plane's rows are N bytes: TMA wants them 16-byte aligned
    return w4a8_tc_int4_supported(xq, qw, s16, out, M, N, K) && N % 16 == 0 && w4a8_aligned(qh, 16);
}

w4a8_status w4a8_launch_int5_tc(const uint8_t *xq, const float *x_scale, const int32_t *qw, const uint8_t *qh,
                                const uint16_t *s16, const uint8_t *zeros, uint16_t *out, int64_t M, int64_t N,
                                int64_t K, void *workspace, int, cudaStream_t stream)
{
    if (zeros == nullptr && w4a8_int4_pf_takes(M, true))
        return w4a8_launch_int4_pf(xq, x_scale, qw, qh, s16, out, M, N, K, workspace, stream);
    const Cfg c = w4a8::tci::choose(M, N, K);
    Params prm;
    if (!make_params(prm, c, x_scale, s16, out, M, N, K, workspace)) return W4A8_ERR_CUDA;
    prm.z5 = zeros;
    // the plane makes each ring fill 8 KB larger than int4's: ring depth 3 / 2 / 2
    if (zeros != nullptr) {
        switch (c.BN) {
        case 16: return launch<16, 3, 3, 4, true, true>(qw, xq, prm, stream, qh);
        case 32: return launch<32, 2, 3, 4, true, true>(qw, xq, prm, stream, qh);
        default: return launch<64, 2, 3, 4, true, true>(qw, xq, prm, stream, qh);
        }
    }
    switch (c.BN) {
    case 16: return launch<16, 3, 3, 4, false, true>(qw, xq, prm, stream, qh);
    case 32: return launch<32, 2, 3, 4, false, true>(qw, xq, prm, stream, qh);
    default: return launch<64, 2, 3, 4, false, true>(qw, xq, prm, stream, qh);
    }
}
