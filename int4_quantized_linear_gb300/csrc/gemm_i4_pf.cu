// gemm_i4_pf.cu -- tensor-core (tcgen05, sm_103a) int4 / int5 group-128 W4A8 GEMM, prefill tiling.
//
// "radiance_autoround.py", module docstring and _exact_ref: symmetric int4 weights, one fp16 scale
// per 128 input channels and output column, zero point 8, per-token fp8 (e4m3) activations:
//   out[m,n] = bf16( x_scale[m] * sum_g s[g,n] * sum_{k in g} e4m3(xq[m,k]) * (c[k,n] - 8) ).
// "vllm-radiance (MXFP4)", section "int5 (W5A8)": the same with 5-bit codes, value c - 16.
//
// The decode kernel (gemm_i4_tc.cu) is built for a few tokens: 16-64-token tiles, so every weight
// tile is converted once per token tile and the zero point rides on extra MMAs.  At prefill sizes
// that spends the tensor pipe and the converters on work that does not scale with the tokens.
// This kernel is the prefill counterpart:
//
//   * tiles of 128 output columns (the MMA M, one per tensor-memory lane) x 256 tokens (the MMA
//     N, the largest single-CTA instruction), so a converted weight k-tile feeds 256 tokens;
//   * the operand holds (c - 8) * 2^-9 (int5: (c - 16) * 2^-9), exact in e4m3, so the zero point
//     costs no MMAs: sum_k (c_k - 8) 2^-9 x_k is one kind::f8f6f4 product (wcodes.cuh);
//   * TMA brings the checkpoint words as stored ([16 word rows x 128 columns] per k-tile, and
//     int5's fifth-bit bytes beside them) into a ring of their own, fed by a producer warp of its
//     own, so the converters never wait on an L2 round trip; they write the swizzled operand tile;
//   * a k-tile is one group, so every k-tile's four MMAs (K = 32 each) go to a fresh accumulator
//     of 256 columns; two of them fill tensor memory and alternate;
//   * eight promotion warps (two per tensor-memory lane quarter, 128 token columns each) read a
//     finished group accumulator and add s[g,n] * 512 * partial into 128 fp32 registers per
//     thread, loading the next 32 columns from tensor memory while they add the last 32; they
//     take registers from the other roles with setmaxnreg;
//   * one tcgen05.commit per k-tile: its barrier tells the producer that the activation slot is
//     free, the converters that the operand tile is free and the promotion warps that the group
//     accumulator is complete;
//   * work split, stream-K fix-up (last contributor adds the fp32 partials in CTA order), bounded
//     waits and the gate warp follow the other tensor-core kernels.
//
// Warp roles: 0 TMA producer (activations), 1 TMEM allocator + MMA issuer, 2 gate, 3 TMA producer
// (checkpoint words) (warpgroup 0);
// 4-7 converters (warpgroup 1); 8-15 promotion and epilogue (warpgroups 2 and 3).
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "dispatch.h"
#include "tc_host.cuh"
#include "tc_ptx.cuh"
#include "tc_sched.cuh"
#include "wcodes.cuh"

namespace w4a8 {
namespace tcp {

using namespace tcs;
using tci::i4x8_to_signed_bytes;
using tci::i5x8_to_signed_bytes;

constexpr int NUM_THREADS = 512;  // 16 warps
constexpr int BN = 256;           // tokens per tile
constexpr int MMA_WARP = 1;
constexpr int GATE_WARP = 2;
constexpr int WORD_WARP = 3;      // producer of the checkpoint-word ring
constexpr int CONV_WARP0 = 4;     // warps 4-7
constexpr int EPI_WARP0 = 8;      // warps 8-15: lane quarter warp & 3, token half (warp >> 2) & 1
constexpr int XK = 2;             // k-tiles per activation fill (256 contiguous bytes per token row)
constexpr int US = 2;             // activation ring fills
constexpr int NB = 2;             // group accumulators of BN columns in tensor memory
constexpr int ND = 4;             // k-tile completion barriers
// checkpoint-word ring slots (one k-tile each) and converted operand tiles: int5's slots carry
// the fifth-bit plane too, so it keeps one operand tile fewer
template <bool I5>
struct Depth {
    static constexpr int RS = I5 ? 4 : 3;
    static constexpr int NA = 2;
    static constexpr int CHUNK = I5 ? 16 : 32;  // tokens per output store (int4 has the room for 32)
};
static_assert(ND >= US * XK && ND >= 3 && ND >= NB, "completion barriers");
constexpr int GATE_BARRIER = 2;   // gate warp + MMA warp
constexpr int EPI_BARRIER = 3;    // the eight promotion warps
// Registers per thread after the split (warpgroups 0, 1, then 2 and 3); the kernel is launched
// with 128 per thread (the host checks), and the split never asks for more than that in all.
// 56 / 80 / 184 is the split at which neither the int4 nor the int5 build spills (40 / 64 / 200
// spilled ~48 bytes per thread, and with shared memory filling the L1 array a spill reload is
// an L2 round trip).
template <bool I5>
struct Regs {
    static constexpr int CTRL = 56;
    static constexpr int CONV = 80;
    static constexpr int EPI = 184;
    static_assert(128 * (CTRL + CONV + 2 * EPI) <= NUM_THREADS * 128, "register split");
};

enum : unsigned { ST_TIMEOUT_PRODUCER = 1, ST_TIMEOUT_GATE = 2, ST_TIMEOUT_CONV = 4, ST_TIMEOUT_EPI = 8 };

struct Params {
    const int32_t *qw;     // [K/8, N] checkpoint words
    const uint8_t *qh;     // int5: [K/8, N] fifth-bit plane
    const uint16_t *s16;   // [K/128, N] fp16 group scales
    const float *xs;       // [M] per-token scale
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
// records clock64() per k-tile i < TRACE_N: 0 activations issued, 1 words issued, 2 words seen
// by the converters, 3 operand tile written, 4 MMAs released by the gate, 5 group accumulator
// seen by the promotion (warp 8), 6 released by warp 8, 7 released by warp 12, 8-10 the gate past
// its waits for the group accumulator, the operand tile and the activations (in the order 10, 9, 8),
// 11 the tile's output issued, 12 the promotion warps done with the tile (warp 8, indexed by the
// k-tile that ended the tile), 13 warp 8 starting a tile (indexed by its first k-tile).
constexpr int TRACE_N = 512;
__device__ __forceinline__ void trace_ev(const Params &p, int ev, int i)
{
#ifdef W4A8_TRACE
    if (p.trace != nullptr && blockIdx.x == 0 && i < TRACE_N) p.trace[ev * TRACE_N + i] = (unsigned long long)clock64();
#endif
}

// Shared memory: the activation ring, the checkpoint-word ring, the converted operand tiles, two
// output staging buffers per token half, the tile's token scales, then barriers and flags.
template <bool I5>
struct Layout {
    static constexpr int RS = Depth<I5>::RS, NA = Depth<I5>::NA;
    static constexpr int X_TILE = BN * 128;      // [256 tokens][128 k] e4m3, 128-byte swizzle
    static constexpr int X_FILL = XK * X_TILE;
    static constexpr int A_TILE = BM * 128;      // [128 columns][128 k] e4m3, 128-byte swizzle
    static constexpr int STAGE_BYTES = Depth<I5>::CHUNK * 32 * 2;  // [CHUNK tokens][32 columns] bf16, per warp and buffer
    static constexpr int W_TILE = 16 * BM * 4;     // [16 word rows][128 columns] int32
    static constexpr int H_TILE = I5 ? 16 * BM : 0;  // [16 rows][128 columns] fifth-bit bytes
    static constexpr int R_SLOT = W_TILE + H_TILE;
    static constexpr int X_OFF = 0;
    static constexpr int R_OFF = X_OFF + US * X_FILL;
    static constexpr int A_OFF = R_OFF + RS * R_SLOT;
    static constexpr int STAGE_OFF = A_OFF + NA * A_TILE;
    static constexpr int XS_OFF = STAGE_OFF + 16 * STAGE_BYTES;  // 8 promotion warps x 2 buffers
    static constexpr int BAR_OFF = XS_OFF + BN * 4;
    static constexpr int TOTAL = BAR_OFF + 256 + 1024;  // + alignment slack
    static constexpr int TMEM_COLS = NB * BN;    // 512
    static_assert(TOTAL <= 232448, "shared memory");
    static_assert(8 * (US + 2 * RS + ND + NA + NB + 1) + 32 <= 256, "barrier area");
    static_assert(X_TILE % 1024 == 0 && A_TILE % 1024 == 0 && A_OFF % 1024 == 0, "swizzled tiles");
};


// 32 lanes x 32 consecutive 32-bit columns -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

template <bool I5>
__global__ void __launch_bounds__(NUM_THREADS, 1)
int4_pf_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_q,
               const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_out,
               const Params p)
{
    using L = Layout<I5>;
    constexpr int RS = L::RS, NA = L::NA;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *x_full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);  // activation slot landed
    uint64_t *r_full = x_full + US;    // checkpoint words landed
    uint64_t *r_empty = r_full + RS;   // checkpoint words read by the converters
    uint64_t *done = r_empty + RS;     // a k-tile's MMAs finished (slot, tile and group released)
    uint64_t *a_full = done + ND;      // converted operand tile written
    uint64_t *g_empty = a_full + NA;   // group accumulator promoted
    uint64_t *mma_done = g_empty + NB;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *last_flag = reinterpret_cast<int *>(tmem_slot + 2);
    int *issued = reinterpret_cast<int *>(tmem_slot + 3);    // activation loads issued
    int *r_issued = reinterpret_cast<int *>(tmem_slot + 4);  // word loads issued

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const Sched sched(cta, p.Gsk, p.RU, p.D, p.R, p.U);
    const int n_k = 4 * sched.n_units;  // k-tiles (= groups) this CTA processes

    if (threadIdx.x == 0) {
        for (int s = 0; s < US; ++s) tc::mbar_init(&x_full[s], 1);        // producer expect_tx
        for (int s = 0; s < RS; ++s) {
            tc::mbar_init(&r_full[s], 1);                                   // word producer expect_tx
            tc::mbar_init(&r_empty[s], 4);                                  // the four converter warps
        }
        for (int d = 0; d < ND; ++d) tc::mbar_init(&done[d], 1);          // tcgen05.commit
        for (int a = 0; a < NA; ++a) tc::mbar_init(&a_full[a], 4);        // the four converter warps
        for (int b = 0; b < NB; ++b) tc::mbar_init(&g_empty[b], 8);       // the eight promotion warps
        tc::mbar_init(mma_done, 1);
        *abort_flag = 0;
        *last_flag = 0;
        *issued = 0;
        *r_issued = 0;
        tc::fence_mbar_init();
        tc::tma_prefetch_desc(&tmap_x);
        tc::tma_prefetch_desc(&tmap_q);
        if (I5) tc::tma_prefetch_desc(&tmap_h);
        if (p.tma_out) tc::tma_prefetch_desc(&tmap_out);
    }
    if (warp == MMA_WARP) {
        tc::tmem_alloc(tmem_slot, L::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // programmatic dependent launch: global memory only after the previous kernel completed
    tc::grid_dependency_wait();
    tc::grid_dependents_launch();

    // tile coordinates of k-tile position i: weight column base n0, token base m0, k-tile kt
    auto coords = [&](int i, int &n0, int &m0, int &kt) {
        const long long u = sched.unit_at(i / 4);
        const int t = (int)div_nonneg(u, p.U);
        kt = (int)(u - (long long)t * p.U) * 4 + (i & 3);
        n0 = (int)((unsigned)t / (unsigned)p.m_tiles) * BM;
        m0 = (int)((unsigned)t % (unsigned)p.m_tiles) * BN;
    };

    if (warp < CONV_WARP0) {
        tc::regs_dec<Regs<I5>::CTRL>();
        if (warp == 0) {
            // -------------------------------------------------------- TMA producer: activations
            if (lane == 0) {
                const uint64_t keep = tc::make_policy_evict_last();  // re-read by the other column tiles
                // fill f holds k-tiles XK f .. XK f + XK - 1 (a unit holds a whole number of fills);
                // its slot is free once the last k-tile of fill f - US is done
                for (int f = 0; f < n_k / XK && !*abort_flag; ++f) {
                    const int s = f % US, last = XK * (f - US) + XK - 1;
                    if (f >= US && wait_or_fail(&done[last % ND], (last / ND) & 1, abort_flag, p.status,
                                                ST_TIMEOUT_PRODUCER, f))
                        break;
                    int n0, m0, kt;
                    coords(XK * f, n0, m0, kt);
                    tc::mbar_arrive_expect_tx(&x_full[s], L::X_FILL);
                    tc::tma_load_3d_hint(smem + L::X_OFF + s * L::X_FILL, &tmap_x, &x_full[s], 0, m0, kt, keep);
                    *issued = f + 1;
                    trace_ev(p, 0, XK * f);
                }
            }
            __syncwarp();
        } else if (warp == WORD_WARP) {
            // -------------------------------------------------------- TMA producer: checkpoint words
            if (lane == 0) {
                for (int i = 0; i < n_k && !*abort_flag; ++i) {
                    const int s = i % RS;
                    if (wait_or_fail(&r_empty[s], ((i / RS) & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER, i))
                        break;
                    int n0, m0, kt;
                    coords(i, n0, m0, kt);
                    uint8_t *dst = smem + L::R_OFF + s * L::R_SLOT;
                    tc::mbar_arrive_expect_tx(&r_full[s], L::R_SLOT);
                    tc::tma_load_2d(dst, &tmap_q, &r_full[s], n0, 16 * kt);
                    if constexpr (I5) tc::tma_load_2d(dst + L::W_TILE, &tmap_h, &r_full[s], n0, 16 * kt);
                    *r_issued = i + 1;
                    trace_ev(p, 1, i);
                }
            }
            __syncwarp();
        } else if (warp == MMA_WARP || warp == GATE_WARP) {
            // -------------------------------------------------------- MMA issuer and its gate
            // The gate waits (group accumulator free, operand tile converted, activations landed)
            // and releases the MMA warp through a named barrier once per k-tile; the MMA thread
            // touches no shared memory while its MMAs run.
            const bool gate = (warp == GATE_WARP);
            if (!gate) tc::tc_fence_after();
            const uint32_t idesc = tc::idesc_f8f6f4(0, 0, BM, BN);
            for (int i = 0; i < n_k; ++i) {
                const int xf = i / XK, s = xf % US, a = i % NA, b = i % NB;
                if (gate && lane == 0) {
                    // the activations and the operand tile are usually ready long before the group
                    // accumulator comes free, so that wait goes last: once it passes, the MMAs are
                    // released at once
                    if (!*abort_flag) wait_or_fail(&x_full[s], (xf / US) & 1, abort_flag, p.status, ST_TIMEOUT_GATE, i);
                    trace_ev(p, 10, i);
                    if (!*abort_flag) wait_or_fail(&a_full[a], (i / NA) & 1, abort_flag, p.status, ST_TIMEOUT_GATE, i);
                    trace_ev(p, 9, i);
                    if (!*abort_flag)
                        wait_or_fail(&g_empty[b], ((i / NB) & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_GATE, i);
                    trace_ev(p, 8, i);
                }
                const bool aborted = tc::named_bar_or(GATE_BARRIER, 64, gate && *abort_flag);
                if (aborted) break;
                if (!gate && lane == 0) {
                    trace_ev(p, 4, i);
                    tc::tc_fence_after();
                    const uint32_t aa = tc::smem_u32(smem + L::A_OFF + a * L::A_TILE);
                    const uint32_t xa = tc::smem_u32(smem + L::X_OFF + s * L::X_FILL + (i % XK) * L::X_TILE);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_f8f6f4(tmem + b * BN, tc::smem_desc(aa + 32 * kk, 16, 1024, 2),
                                       tc::smem_desc(xa + 32 * kk, 16, 1024, 2), idesc, kk > 0 ? 1u : 0u);
                    tc::tc_commit(&done[i % ND]);
                }
                __syncwarp();
            }
            if (!gate && lane == 0) tc::tc_commit(mma_done);  // teardown waits on it before freeing TMEM
            __syncwarp();
        }
    } else if (warp < EPI_WARP0) {
        tc::regs_dec<Regs<I5>::CONV>();
        // ------------------------------------------------------------ converters (4-7)
        // Thread = one weight column r of the tile: it reads the column's 16 words of a k-tile (int5:
        // and their 16 fifth-bit bytes) from the word ring (consecutive columns are consecutive
        // words: no bank conflicts) and writes the 128 e4m3 codes of (c - 8) * 2^-9 (int5:
        // (c - 16) * 2^-9) as eight 16-byte chunks at their swizzled places in row r of the
        // operand tile.
        const int r = 32 * (warp - CONV_WARP0) + lane;
        for (int i = 0; i < n_k; ++i) {
            const int s = i % RS, a = i % NA;
            if (warp_wait(&r_full[s], (i / RS) & 1, abort_flag, p.status, ST_TIMEOUT_CONV, i, lane)) break;
            if (r == 0) trace_ev(p, 2, i);
            // the operand tile is free once k-tile i - NA's MMAs are done
            if (i >= NA && warp_wait(&done[(i - NA) % ND], ((i - NA) / ND) & 1, abort_flag, p.status,
                                     ST_TIMEOUT_CONV, i, lane))
                break;
            const uint8_t *raw = smem + L::R_OFF + s * L::R_SLOT;
            uint32_t wv[16], hv[I5 ? 16 : 1];
#pragma unroll
            for (int j = 0; j < 16; ++j) wv[j] = reinterpret_cast<const uint32_t *>(raw)[j * BM + r];
            if constexpr (I5) {
#pragma unroll
                for (int j = 0; j < 16; ++j) hv[j] = raw[L::W_TILE + j * BM + r];
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&r_empty[s]);  // the words are in registers
            uint8_t *dst = smem + L::A_OFF + a * L::A_TILE + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {  // chunk c = k 16c .. 16c + 15 = words 2c, 2c + 1
                uint2 lo, hi;
                if constexpr (I5) {
                    lo = i5x8_to_signed_bytes(wv[2 * c], hv[2 * c]);
                    hi = i5x8_to_signed_bytes(wv[2 * c + 1], hv[2 * c + 1]);
                } else {
                    lo = i4x8_to_signed_bytes(wv[2 * c]);
                    hi = i4x8_to_signed_bytes(wv[2 * c + 1]);
                }
                *reinterpret_cast<uint4 *>(dst + ((c ^ (r & 7)) << 4)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
            }
            tc::fence_proxy_async_smem();  // generic writes -> visible to the tensor core
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&a_full[a]);
            if (r == 0) trace_ev(p, 3, i);
        }
    } else {
        tc::regs_inc<Regs<I5>::EPI>();
        // ------------------------------------------------------------ promotion and epilogue (8-15)
        // Warp w reads tensor-memory lanes 32q..32q+31 (q = w & 3: weight columns n0 + 32q + lane)
        // and token columns 128h..128h+127 of the tile (h = (w >> 2) & 1).
        const int q = warp & 3, h = (warp >> 2) & 1;
        const int r = 32 * q + lane;
        float *xs_s = reinterpret_cast<float *>(smem + L::XS_OFF) + 128 * h;
        int ck = 0;  // output chunks emitted by this half (staging buffer rotation)
        // Write 16 token columns (tile columns c0..c0+15 of this half) of this thread's weight
        // column: each warp through a [CHUNK tokens][32 columns] bf16 stage of its own (two of
        // them, alternating), filled 16 tokens at a time, and one TMA store per CHUNK tokens issued
        // by its lane 0 -- no barrier across warps -- or plain stores.  `last`: no more tokens
        // follow in this half, so a partly filled stage goes out (its unwritten rows are tokens at
        // or past M, which the store clips).
        constexpr int CHUNK = Depth<I5>::CHUNK;
        auto emit = [&](const float (&o)[16], int c0, int m0, int n0, bool last) {
            const int n = n0 + r;
            if (p.tma_out) {
                const int sub = (c0 / 16) % (CHUNK / 16);  // which 16 tokens of the stage
                uint16_t *stg = reinterpret_cast<uint16_t *>(smem + L::STAGE_OFF +
                                                             (2 * (warp - EPI_WARP0) + (ck & 1)) * L::STAGE_BYTES);
                if (sub == 0 && ck >= 2) {  // the store that last used this buffer has read it
                    if (lane == 0) tc::bulk_wait_group_read<1>();
                    __syncwarp();
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) stg[(16 * sub + j) * 32 + lane] = float_to_bf16_bits(o[j]);
                if (sub == CHUNK / 16 - 1 || last) {
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && n0 + 32 * q < p.N) {  // (a warp wholly past the last column stores nothing)
                        tc::tma_store_2d_hint(&tmap_out, stg, n0 + 32 * q, m0 + c0 - 16 * sub,
                                              tc::make_policy_evict_first());
                        tc::bulk_commit_group();
                    }
                    ++ck;
                }
            } else if (n < p.N) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (m0 + c0 + j < p.M) tc::st_cg_u16(p.out + (size_t)(m0 + c0 + j) * p.N + n, float_to_bf16_bits(o[j]));
            }
        };
        // group scales of one unit (4 k-tiles) for this thread's column, times 2^9 (the operand
        // codes are (c - 8) * 2^-9), fetched a unit ahead
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
        float sc_cur[4] = {0.0f, 0.0f, 0.0f, 0.0f}, sc_nxt[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        unit_scales(0, sc_nxt);
        int i = 0;  // k-tile position, in the order the MMAs run
        for (int seg = 0; seg < sched.S; ++seg) {
            long long u, ue;
            sched.seg_units(seg, u, ue);
            const int t = (int)div_nonneg(u, p.U);
            const long long t_lo = (long long)t * p.U, t_hi = t_lo + p.U;
            const bool whole = (u == t_lo) && (ue == t_hi);
            const int n0 = (t / p.m_tiles) * BM, m0 = (t % p.m_tiles) * BN;
            // this half's token scales: loaded now, stored to shared memory after the tile's k-tiles
            // (no wait on the load at the start of the tile; the previous tile's readers are done)
            const float xs_r = (m0 + 128 * h + r < p.M) ? __ldg(p.xs + m0 + 128 * h + r) : 0.0f;
            float acc[128];
#pragma unroll
            for (int c = 0; c < 128; ++c) acc[c] = 0.0f;
            if (threadIdx.x == EPI_WARP0 * 32) trace_ev(p, 13, i);
            bool gave_up = false;
            for (const int i_end = i + 4 * (int)(ue - u); i < i_end; ++i) {
                const int b = i % NB, jj = i & 3;
                if (jj == 0) {
#pragma unroll
                    for (int z = 0; z < 4; ++z) sc_cur[z] = sc_nxt[z];
                    unit_scales(i / 4 + 1, sc_nxt);
                }
                int w = 0;
                if (lane == 0) w = tc::mbar_wait(&done[i % ND], (i / ND) & 1, abort_flag, WAIT_BUDGET);
                w = __shfl_sync(0xffffffffu, w, 0);
                if (w) {
                    if (lane == 0) {
                        if (w == 1) fail(p.status, ST_TIMEOUT_EPI, &done[i % ND], i);
                        *abort_flag = 1;
                    }
                    gave_up = true;
                    break;
                }
                tc::tc_fence_after();
                if (threadIdx.x == EPI_WARP0 * 32) trace_ev(p, 5, i);
                const float s = jj == 0 ? sc_cur[0] : jj == 1 ? sc_cur[1] : jj == 2 ? sc_cur[2] : sc_cur[3];
                const uint32_t tb = tmem + b * BN + 128 * h + ((32u * q) << 16);
                // two 32-column buffers: the next load is in flight while the last one is added
                uint32_t va[32], vb[32];
                tmem_ld32(tb, va);
                tc::tmem_ld_wait();
                tmem_ld32(tb + 32, vb);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[j] = fmaf(s, __uint_as_float(va[j]), acc[j]);
                tc::tmem_ld_wait();
                tmem_ld32(tb + 64, va);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[32 + j] = fmaf(s, __uint_as_float(vb[j]), acc[32 + j]);
                tc::tmem_ld_wait();
                tmem_ld32(tb + 96, vb);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[64 + j] = fmaf(s, __uint_as_float(va[j]), acc[64 + j]);
                tc::tmem_ld_wait();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&g_empty[b]);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[96 + j] = fmaf(s, __uint_as_float(vb[j]), acc[96 + j]);
                if (threadIdx.x == EPI_WARP0 * 32) trace_ev(p, 6, i);
                if (threadIdx.x == (EPI_WARP0 + 4) * 32) trace_ev(p, 7, i);
            }
            xs_s[r] = xs_r;
            // all eight warps leave together if any gave up (this also publishes xs_s)
            if (tc::named_bar_or(EPI_BARRIER, 256, gave_up)) break;
            if (threadIdx.x == EPI_WARP0 * 32) trace_ev(p, 12, i - 1);
            if (whole) {
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 16) {
                    if (m0 + 128 * h + c0 < p.M) {
                        float o[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) o[j] = acc[c0 + j] * xs_s[c0 + j];
                        emit(o, 128 * h + c0, m0, n0, c0 + 16 >= 128 || m0 + 128 * h + c0 + 16 >= p.M);
                    }
                }
            } else {
                // stream-K: store this CTA's fp32 partial; the last contributor adds all in CTA order
                float *slot = p.partials + ((size_t)cta * 2 + (t == sched.t_first ? 0 : 1)) * (size_t)(BM * BN);
#pragma unroll
                for (int c = 0; c < 128; ++c) tc::st_cg_f32(slot + (128 * h + c) * BM + r, acc[c]);
                const int c_first = unit_owner(t_lo, p.RU, p.Gsk);
                const int c_last = unit_owner(t_hi - 1, p.RU, p.Gsk);
                // every partial store happens before one thread's acq_rel arrival (release); the last
                // arrival's acquire makes every contributor's partial visible to it
                tc::named_bar_sync(EPI_BARRIER, 256);
                if (threadIdx.x == EPI_WARP0 * 32) {
                    const int old = tc::atomic_add_acq_rel_gpu(p.counters + t, 1);
                    *last_flag = (old == c_last - c_first);
                }
                tc::named_bar_sync(EPI_BARRIER, 256);
                if (*last_flag) {
                    const int m_cnt = min(128, p.M - m0 - 128 * h);
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
                                const float *src = p.partials + ((size_t)c * 2 + sl) * (size_t)(BM * BN) +
                                                   (128 * h + c0) * BM + r;
#pragma unroll
                                for (int j = 0; j < 16; ++j) v[cc][j] = __ldcg(src + j * BM);
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
                        emit(sum, 128 * h + c0, m0, n0, c0 + 16 >= m_cnt);
                    }
                    if (threadIdx.x == EPI_WARP0 * 32) p.counters[t] = 0;
                }
                tc::named_bar_sync(EPI_BARRIER, 256);  // last_flag is reused by the next tile
            }
            if (threadIdx.x == EPI_WARP0 * 32) trace_ev(p, 11, i - 1);
        }
        if (lane == 0) tc::bulk_wait_group_all();  // output stores done before shared memory goes away
    }

    tc::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        int zero = 0;
        if (*abort_flag) {  // drain: TMA copies issued but not waited for
            for (int f = max(0, *issued - US); f < *issued; ++f)
                if (tc::mbar_wait(&x_full[f % US], (f / US) & 1, &zero, DRAIN_BUDGET)) break;
            for (int f = max(0, *r_issued - RS); f < *r_issued; ++f)
                if (tc::mbar_wait(&r_full[f % RS], (f / RS) & 1, &zero, DRAIN_BUDGET)) break;
        }
        tc::mbar_wait(mma_done, 0, &zero, WAIT_BUDGET);  // every MMA finished before TMEM is freed
    }
    __syncthreads();
    if (warp == MMA_WARP) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// ------------------------------------------------------------------------------- host side

struct Cfg {
    int m_tiles, n_tiles, U;
    SkSplit k;
};

static Cfg choose(int64_t M, int64_t N, int64_t K)
{
    Cfg c;
    c.n_tiles = (int)((N + BM - 1) / BM);
    c.m_tiles = (int)((M + BN - 1) / BN);
    c.U = (int)(K / 512);
    c.k = sk_split((long long)c.n_tiles * c.m_tiles, c.U, tch::num_sms());
    return c;
}

static size_t partial_bytes(const Cfg &c)
{
    const size_t b = (size_t)c.k.G * 2 * BM * BN * 4;
    return (b + 255) / 256 * 256;
}

// The register split assumes the kernel is launched with 128 registers per thread; a build
// that gave it fewer would leave setmaxnreg.inc waiting for registers that do not exist, so such
// a build never runs this kernel (the callers then keep the 64-token kernel).
template <bool I5>
static bool regs_ok()
{
    static std::atomic<int> state{0};  // 0 unknown, 1 yes, 2 no
    int s = state.load(std::memory_order_acquire);
    if (s == 0) {
        cudaFuncAttributes fa;
        const bool ok = cudaFuncGetAttributes(&fa, int4_pf_kernel<I5>) == cudaSuccess &&
                        fa.maxThreadsPerBlock >= NUM_THREADS &&
                        128 * (Regs<I5>::CTRL + Regs<I5>::CONV + 2 * Regs<I5>::EPI) <= NUM_THREADS * fa.numRegs;
        s = ok ? 1 : 2;
        state.store(s, std::memory_order_release);
    }
    return s == 1;
}

template <bool I5>
static w4a8_status launch(const uint8_t *xq, Params prm, cudaStream_t stream)
{
    using L = Layout<I5>;
    CUtensorMap tx, tq, th, tout;
    memset(&tout, 0, sizeof(tout));
    memset(&th, 0, sizeof(th));
    // checkpoint words [K/8 rows][N columns] int32 and (int5) the plane [K/8][N] bytes: boxes of
    // one k-tile's 16 rows x 128 columns
    if (!tch::tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_INT32, prm.qw, prm.K / 8, prm.N, (uint64_t)prm.N * 4, 16, BM,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
        (I5 && !tch::tmap_2d(&th, CU_TENSOR_MAP_DATA_TYPE_UINT8, prm.qh, prm.K / 8, prm.N, (uint64_t)prm.N, 16, BM,
                             CU_TENSOR_MAP_SWIZZLE_NONE)))
        return W4A8_ERR_CUDA;
    prm.tma_out = (prm.N % 8 == 0) && w4a8_aligned(prm.out, 16) &&
                  tch::tmap_2d(&tout, CU_TENSOR_MAP_DATA_TYPE_UINT16, prm.out, prm.M, prm.N, (uint64_t)prm.N * 2,
                               Depth<I5>::CHUNK, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
    // activations as [k-tile][token][128 bytes], XK k-tiles of 256 tokens per box
    if (!tch::tmap_3d_ktiles(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, prm.M, prm.K, 128, prm.K / 128, BN, XK))
        return W4A8_ERR_CUDA;
    auto kern = int4_pf_kernel<I5>;
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
    if (cudaLaunchKernelEx(&cfg, kern, tx, tq, th, tout, prm) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return w4a8_launch_status();
}

}  // namespace tcp
}  // namespace w4a8

using namespace w4a8::tcp;

bool w4a8_int4_pf_takes(int64_t M, bool int5)
{
    if (M <= W4A8_INT4_PF_MIN_M) return false;
    return int5 ? regs_ok<true>() : regs_ok<false>();
}

size_t w4a8_int4_pf_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (K % 512 != 0 || K <= 0 || M <= 0 || N <= 0) return 0;
    const Cfg c = choose(M, N, K);
    return W4A8_COUNTER_BYTES + partial_bytes(c);
}

w4a8_status w4a8_launch_int4_pf(const uint8_t *xq, const float *x_scale, const int32_t *qw, const uint8_t *qh,
                                const uint16_t *s16, uint16_t *out, int64_t M, int64_t N, int64_t K, void *workspace,
                                cudaStream_t stream)
{
    const Cfg c = choose(M, N, K);
    Params prm;
    prm.qw = qw;
    prm.qh = qh;
    prm.s16 = s16;
    prm.xs = x_scale;
    prm.out = out;
    prm.counters = static_cast<int *>(workspace);
    prm.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + W4A8_COUNTER_BYTES);
    prm.status = w4a8_device_status_ptr();
    if (!prm.status || c.k.G > W4A8_MAX_COUNTERS) return W4A8_ERR_CUDA;
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
    return qh ? launch<true>(xq, prm, stream) : launch<false>(xq, prm, stream);
}
