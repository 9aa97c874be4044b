// gemm_tc.cu -- tensor-core (tcgen05, sm_103a) MXFP4 W4A8 GEMM, persistent stream-K.
//
// "vllm-radiance (MXFP4)", "The W4A8 fp8-WMMA kernel": fp8 (e4m3) activations times e2m1
// weights with the e8m0 block scale folded into the matrix instruction; a prefill tiling and a
// decode tiling; the decode K-splits are reduced in place by the last CTA to arrive, with no
// second launch and a result independent of arrival order.  The pages' kernel is an RDNA4 WMMA
// design; this one is built for Blackwell:
//
//   * swap-AB: the weights are the MMA "M" operand (128 weight rows per tile) and the tokens the
//     "N" operand (16..256), so a decode batch of 1-64 tokens still fills the instruction;
//   * tcgen05.mma kind::mxf8f6f4 block_scale.scale_vec::1X: A = e2m1 weights with their ue8m0
//     scale per 32 along K, B = e4m3 activations with a unit scale (0x7F), fp32 accumulators in
//     tensor memory; the per-token scale multiplies in the epilogue;
//   * TMA brings the packed weights (64 bytes per row per k-tile), the activations (128-byte
//     swizzle) and, once per 4 k-tiles, a [128 x 16-byte] tile of weight scales.  A converter
//     warpgroup rewrites each packed weight tile into the form the instruction reads for 4-bit
//     operands -- 16 codes in the low 8 bytes of each 16-byte slot, 128-byte swizzle -- and widens
//     each row's 4-byte scale word into a 16-byte row, which tcgen05.cp copies to tensor memory
//     (lane r of each scale column then holds row r's word).  (TMA can do the 4-bit padding itself
//     with its 16U4_ALIGN16B type, but measured on GB300 that path moves only about 16 GB/s of
//     packed data per SM, far below an SM's share of HBM bandwidth.);
//   * persistent stream-K: one CTA per SM walks a contiguous range of (tile, 4-k-tile unit)
//     work, so the TMA ring never drains between tiles and every SM gets the same number of
//     units; a tile whose K range is split between CTAs is finished by the last contributor,
//     which adds the fp32 partials in CTA order;
//   * two accumulator buffers in tensor memory (one for 256-token tiles) let the MMAs of the next
//     tile run while the epilogue drains the previous one;
//   * warp roles: 0 TMA producer, 1 TMEM allocator + MMA issuer, 2-5 converters, 6-9 epilogue
//     (each epilogue warp reads the TMEM lane quarter its warp index selects).
//
// Every mbarrier wait is bounded; a wait that runs out sets a bit in the library's device status
// word and the CTA winds down (draining what it started) instead of hanging.
#include "common.cuh"
#include "dispatch.h"
#include "tc_host.cuh"
#include "tc_ptx.cuh"

namespace w4a8 {
namespace tcg {

constexpr int BM = 128;            // weight rows per tile (MMA M)
constexpr int BK = 128;            // K elements per pipeline stage (one k-tile)
constexpr int NUM_THREADS = 320;   // 10 warps
constexpr int CONV_WARP0 = 2;      // warps 2-5
constexpr int EPI_WARP0 = 6;       // warps 6-9
constexpr long long WAIT_BUDGET = 1ll << 29;  // clock cycles (a quarter second or so)
constexpr long long DRAIN_BUDGET = 1ll << 24;

enum : unsigned { ST_TIMEOUT_PRODUCER = 1, ST_TIMEOUT_MMA = 2, ST_TIMEOUT_CONV = 4, ST_TIMEOUT_EPI = 8 };

struct Params {
    const uint8_t *we;     // [N, K/32] e8m0
    const float *xs;       // [M] per-token scale
    uint16_t *out;         // [M, N] bf16
    float *partials;       // [G][2][BN][128] fp32 stream-K partial tiles
    int *counters;         // [tiles] arrival counters, zero between calls
    unsigned int *status;  // device status block
    int M, N, K;
    int m_tiles, n_tiles;
    int U;                 // 4-k-tile units per tile
    long long TU;          // total units
    int G;                 // CTAs
    unsigned long long *trace;  // optional pipeline timeline of CTA 0 (diagnostics), or null
};

// Pipeline timeline (diagnostics): CTA 0 records clock64() per k-tile i < TRACE_N for each event.
constexpr int TRACE_N = 256;
enum { TR_TMA_ISSUED = 0, TR_CONV_DATA, TR_CONV_DONE, TR_MMA_READY, TR_MMA_ISSUED, TR_SLOT_FREED, TR_EVENTS };
__device__ __forceinline__ void trace_ev(const Params &p, int ev, int i)
{
    if (p.trace != nullptr && blockIdx.x == 0 && i < TRACE_N) p.trace[ev * TRACE_N + i] = (unsigned long long)clock64();
}

// Shared memory.  Ring A (depth STAGES) holds what TMA writes for a k-tile: the activation
// tile and the weight tile -- already in the padded 4-bit form when TMA does the padding
// (CONV = false), packed when a converter warpgroup pads it (CONV = true), in which case ring B
// (depth PSTAGES) holds the padded tiles.  Raw scale tiles (4 k-tiles each) have a ring of 2.
template <int BN, int STAGES, int PSTAGES, int ACC_BUFS, bool CONV>
struct Layout {
    static constexpr int X_BYTES = BN * 128;               // BN tokens x 128 K bytes (swizzled)
    static constexpr int W_BYTES = BM * 128;               // padded: 128 rows x 8 slots of 16 bytes
    static constexpr int WP_BYTES = BM * 64;               // packed: 128 rows x 64 bytes
    static constexpr int A_W_BYTES = CONV ? WP_BYTES : W_BYTES;
    static constexpr int B_SLOTS = CONV ? PSTAGES : 0;
    static constexpr int SF_SLOTS = CONV ? PSTAGES : STAGES;  // TMEM scale slots (4 columns each)
    static constexpr int SFR_SLOTS = 2;
    static constexpr int SFR_BYTES = BM * 16;              // 128 rows x 16 bytes = 4 k-tiles
    static constexpr int X_OFF = 0;
    static constexpr int AW_OFF = X_OFF + STAGES * X_BYTES;   // 1024-aligned for the swizzled form
    static constexpr int BW_OFF = AW_OFF + STAGES * A_W_BYTES;
    static constexpr int SFR_OFF = BW_OFF + B_SLOTS * W_BYTES;
    static constexpr int BAR_OFF = SFR_OFF + SFR_SLOTS * SFR_BYTES;
    static constexpr int TOTAL = BAR_OFF + 512 + 1024;  // barriers, flags, alignment slack
    static constexpr int W_TX_BYTES = BM * 64;          // both forms count the packed bytes
    static constexpr int T_SFB = ACC_BUFS * BN;         // TMEM column of the unit B scales
    static constexpr int T_SFA = T_SFB + 8;             // TMEM columns of the A scales
    static constexpr int TMEM_NEED = T_SFA + 4 * SF_SLOTS;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64
                                     : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
    static_assert(TMEM_NEED <= 512, "tensor memory");
    static_assert(TOTAL <= 232448, "shared memory");
    static_assert((X_BYTES % 1024) == 0 && (AW_OFF % 1024) == 0 && (BW_OFF % 1024) == 0, "alignment");
};

// Record a bounded wait that ran out: the role's bit in word 0 of the status block; the first
// such event also leaves its loop index (word 1) and the barrier's raw state (words 2-3).
__device__ __forceinline__ void fail(unsigned int *status, unsigned int bit, uint64_t *bar, int iter)
{
    const unsigned int prev = atomicOr(status, bit);
    if (prev == 0) {
        const uint64_t raw = tc::mbar_raw(bar);
        status[1] = (unsigned int)iter;
        status[2] = (unsigned int)raw;
        status[3] = (unsigned int)(raw >> 32);
    }
}

// First unit of CTA c, and the CTA that owns unit u, for the even split of TU units over G CTAs.
__device__ __forceinline__ long long unit_start(long long c, long long TU, int G) { return c * TU / G; }
__device__ __forceinline__ int unit_owner(long long u, long long TU, int G) { return (int)(((u + 1) * G - 1) / TU); }

// Warp-uniform bounded wait by lane 0; on a timeout or abort the warp records it and returns
// nonzero.
__device__ __forceinline__ int warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         unsigned int *status, unsigned int bit, int iter, int lane)
{
    int w = 0;
    if (lane == 0) {
        w = tc::mbar_wait(bar, parity, abort_flag, WAIT_BUDGET);
        if (w == 1) fail(status, bit, bar, iter);
        if (w) *abort_flag = 1;
    }
    return __shfl_sync(0xffffffffu, w, 0);
}

template <int BN, int STAGES, int PSTAGES, int ACC_BUFS, bool CONV>
__global__ void __launch_bounds__(NUM_THREADS, 1)
mxfp4_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_sf, const Params p)
{
    using L = Layout<BN, STAGES, PSTAGES, ACC_BUFS, CONV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);  // ring A landed (+ scales)
    uint64_t *empty = full + STAGES;                                    // ring A free again
    uint64_t *pfull = empty + STAGES;                                   // ring B converted
    uint64_t *pempty = pfull + PSTAGES;                                 // ring B free again
    uint64_t *sfr_full = pempty + PSTAGES;
    uint64_t *sfr_empty = sfr_full + L::SFR_SLOTS;
    uint64_t *acc_full = sfr_empty + L::SFR_SLOTS;
    uint64_t *acc_empty = acc_full + ACC_BUFS;
    uint64_t *mma_done = acc_empty + ACC_BUFS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *last_flag = reinterpret_cast<int *>(tmem_slot + 2);
    int *consumed = reinterpret_cast<int *>(tmem_slot + 3);
    int *issued = reinterpret_cast<int *>(tmem_slot + 4);
    int *sfr_issued = reinterpret_cast<int *>(tmem_slot + 5);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u_begin = unit_start(cta, p.TU, p.G);
    const long long u_end = unit_start(cta + 1, p.TU, p.G);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // producer expect_tx + 4 scale warps (which also convert, when CONV)
            tc::mbar_init(&full[s], CONV ? 1 : 5);
            // MMA commit (+ the 4 converter warps done with the packed tile, when CONV)
            tc::mbar_init(&empty[s], CONV ? 5 : 1);
        }
        for (int s = 0; s < PSTAGES; ++s) {
            tc::mbar_init(&pfull[s], 4);   // one arrival per converter warp
            tc::mbar_init(&pempty[s], 1);  // tcgen05.commit of the k-tile's MMAs
        }
        for (int r = 0; r < L::SFR_SLOTS; ++r) {
            tc::mbar_init(&sfr_full[r], 1);
            tc::mbar_init(&sfr_empty[r], 4);  // one arrival per scale warp
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            tc::mbar_init(&acc_full[b], 1);   // tcgen05.commit after a tile's last MMA
            tc::mbar_init(&acc_empty[b], 1);  // epilogue finished reading the buffer
        }
        tc::mbar_init(mma_done, 1);
        *abort_flag = 0;
        *last_flag = 0;
        *consumed = 0;
        *issued = 0;
        *sfr_issued = 0;
        tc::fence_mbar_init();
        tc::tma_prefetch_desc(&tmap_w);
        tc::tma_prefetch_desc(&tmap_x);
        tc::tma_prefetch_desc(&tmap_sf);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, L::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Unit scale (2^0) for the activation operand: 0x7F in every byte of the B-scale columns.
    if (warp >= EPI_WARP0) {
        const uint32_t base = tmem + L::T_SFB + ((32u * (warp & 3)) << 16);
        tc::tmem_st4(base, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
        tc::tmem_st4(base + 4, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
        tc::tmem_st_wait();
    }
    tc::tc_fence_before();
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int i = 0, g = 0;
            for (long long u = u_begin; u < u_end && !*abort_flag; ++u, ++g) {
                const int t = (int)(u / p.U), ku = (int)(u - (long long)t * p.U);
                const int n0 = (t / p.m_tiles) * BM, m0 = (t % p.m_tiles) * BN;
                const int rs = g % L::SFR_SLOTS;
                int w = tc::mbar_wait(&sfr_empty[rs], ((g / L::SFR_SLOTS) & 1) ^ 1, abort_flag, WAIT_BUDGET);
                if (w) {
                    if (w == 1) fail(p.status, ST_TIMEOUT_PRODUCER, &sfr_empty[rs], g);
                    *abort_flag = 1;
                    break;
                }
                tc::mbar_arrive_expect_tx(&sfr_full[rs], L::SFR_BYTES);
                tc::tma_load_2d(smem + L::SFR_OFF + rs * L::SFR_BYTES, &tmap_sf, &sfr_full[rs], 16 * ku, n0);
                *sfr_issued = g + 1;
                for (int j = 0; j < 4; ++j, ++i) {
                    const int s = i % STAGES;
                    w = tc::mbar_wait(&empty[s], ((i / STAGES) & 1) ^ 1, abort_flag, WAIT_BUDGET);
                    if (w) {
                        if (w == 1) fail(p.status, ST_TIMEOUT_PRODUCER, &empty[s], i);
                        *abort_flag = 1;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(&full[s], L::W_TX_BYTES + L::X_BYTES);
                    const int k = (4 * ku + j) * BK;
                    // weights: element coordinate k in the 4-bit map, byte coordinate k/2 in the byte map
                    tc::tma_load_2d(smem + L::AW_OFF + s * L::A_W_BYTES, &tmap_w, &full[s], CONV ? k / 2 : k, n0);
                    tc::tma_load_2d(smem + L::X_OFF + s * L::X_BYTES, &tmap_x, &full[s], k, m0);
                    *issued = i + 1;
                    trace_ev(p, TR_TMA_ISSUED, i);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            tc::tc_fence_after();
            int i = 0, seg = 0;
            long long u = u_begin;
            while (u < u_end && !*abort_flag) {
                const int t = (int)(u / p.U);
                const long long ue = min(u_end, (long long)(t + 1) * p.U);
                const int b = seg % ACC_BUFS;
                int w = tc::mbar_wait(&acc_empty[b], ((seg / ACC_BUFS) & 1) ^ 1, abort_flag, WAIT_BUDGET);
                if (w) {
                    if (w == 1) fail(p.status, ST_TIMEOUT_MMA, &acc_empty[b], seg);
                    *abort_flag = 1;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t t_acc = tmem + b * BN;
                bool first = true;
                for (long long k4 = 4 * (ue - u); k4 > 0; --k4, ++i) {
                    const int s = i % STAGES, ps = i % PSTAGES;
                    w = tc::mbar_wait(&full[s], (i / STAGES) & 1, abort_flag, WAIT_BUDGET);
                    if (CONV && !w) w = tc::mbar_wait(&pfull[ps], (i / PSTAGES) & 1, abort_flag, WAIT_BUDGET);
                    if (w) {
                        if (w == 1) fail(p.status, ST_TIMEOUT_MMA, &full[s], i);
                        *abort_flag = 1;
                        break;
                    }
                    *consumed = i + 1;
                    trace_ev(p, TR_MMA_READY, i);
                    tc::tc_fence_after();
                    const int sfs = CONV ? ps : s;
                    const uint32_t sfa = tmem + L::T_SFA + 4 * sfs;
                    const uint32_t wa = CONV ? tc::smem_u32(smem + L::BW_OFF + ps * L::W_BYTES)
                                             : tc::smem_u32(smem + L::AW_OFF + s * L::W_BYTES);
                    const uint32_t xa = tc::smem_u32(smem + L::X_OFF + s * L::X_BYTES);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = tc::smem_desc(wa + 32 * kk, 16, 1024, 2);
                        const uint64_t bd = tc::smem_desc(xa + 32 * kk, 16, 1024, 2);
                        tc::mma_mxf8f6f4(t_acc, ad, bd, tc::idesc_mxf8f6f4(5, 0, BM, BN, kk, 0), sfa,
                                         tmem + L::T_SFB, (first && kk == 0) ? 0u : 1u);
                    }
                    first = false;
                    tc::tc_commit(&empty[s]);
                    if (CONV) tc::tc_commit(&pempty[ps]);
                    trace_ev(p, TR_MMA_ISSUED, i);
                }
                if (w) break;
                tc::tc_commit(&acc_full[b]);
                ++seg;
                u = ue;
            }
            tc::tc_commit(mma_done);  // always: teardown waits on it before freeing TMEM
        }
        __syncwarp();
    } else if (warp < EPI_WARP0) {
        // ------------------------------------------------------------ scale warps (2-5)
        // Each warp owns the TMEM lane quarter q = warp & 3 (weight rows 32q..32q+31) and writes
        // its rows' 4-byte scale word, repeated over the slot's 4 columns, with tcgen05.st.
        // With CONV they also pad the packed weight tile:
        //   packed row r, 16-code chunk c at byte 64r + 8c  ->  padded row r at 128r (rows in
        //   1024-byte groups of 8), chunk c in 16-byte slot c ^ (r & 7), low 8 bytes, zero pad.
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const int ct = threadIdx.x - CONV_WARP0 * 32;  // 0..127 (converter thread)
        int i = 0, g = 0;
        int w = 0;
        for (long long u = u_begin; u < u_end && !w; ++u, ++g) {
            const int rs = g % L::SFR_SLOTS;
            w = warp_wait(&sfr_full[rs], (g / L::SFR_SLOTS) & 1, abort_flag, p.status, ST_TIMEOUT_CONV, g, lane);
            if (w) break;
            const uint8_t *raw = smem + L::SFR_OFF + rs * L::SFR_BYTES;
            for (int j = 0; j < 4; ++j, ++i) {
                const int s = i % STAGES, ps = i % PSTAGES;
                if (CONV) {
                    w = warp_wait(&full[s], (i / STAGES) & 1, abort_flag, p.status, ST_TIMEOUT_CONV, i, lane);
                    if (!w) w = warp_wait(&pempty[ps], ((i / PSTAGES) & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_CONV, i, lane);
                } else {
                    // the scale slot is free once the MMAs that last read it (k-tile i - STAGES) are done
                    w = warp_wait(&empty[s], ((i / STAGES) & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_CONV, i, lane);
                }
                if (w) break;
                if (lane == 0 && warp == CONV_WARP0) trace_ev(p, TR_CONV_DATA, i);
                if (CONV) {
                    const uint8_t *src = smem + L::AW_OFF + s * L::WP_BYTES;
                    uint8_t *dst = smem + L::BW_OFF + ps * L::W_BYTES;
#pragma unroll
                    for (int qq = 0; qq < 8; ++qq) {
                        const int idx = ct + 128 * qq;  // (row, chunk) pair
                        const int r = idx >> 3, c = idx & 7;
                        const uint2 v = *reinterpret_cast<const uint2 *>(src + r * 64 + c * 8);
                        *reinterpret_cast<uint4 *>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = make_uint4(v.x, v.y, 0u, 0u);
                    }
                }
                const uint32_t sw = *reinterpret_cast<const uint32_t *>(raw + row * 16 + 4 * j);
                const int sfs = CONV ? ps : s;
                tc::tmem_st4(tmem + L::T_SFA + 4 * sfs + ((32u * q) << 16), sw, sw, sw, sw);
                tc::tmem_st_wait();
                if (CONV) tc::fence_proxy_async_smem();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (CONV) {
                        tc::mbar_arrive(&pfull[ps]);
                        tc::mbar_arrive(&empty[s]);  // the packed tile is no longer needed
                    } else {
                        tc::mbar_arrive(&full[s]);
                    }
                    if (warp == CONV_WARP0) trace_ev(p, TR_CONV_DONE, i);
                }
            }
            if (w) break;
            if (lane == 0) tc::mbar_arrive(&sfr_empty[rs]);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int first_tile = (int)(u_begin / p.U);
        int seg = 0;
        long long u = u_begin;
        while (u < u_end) {
            const int t = (int)(u / p.U);
            const long long t_lo = (long long)t * p.U, t_hi = t_lo + p.U;
            const long long ue = min(u_end, t_hi);
            const bool whole = (u == t_lo) && (ue == t_hi);
            const int b = seg % ACC_BUFS;
            int w = 0;
            if (lane == 0) w = tc::mbar_wait(&acc_full[b], (seg / ACC_BUFS) & 1, abort_flag, WAIT_BUDGET);
            w = __shfl_sync(0xffffffffu, w, 0);
            if (w) {
                if (lane == 0) {
                    if (w == 1) fail(p.status, ST_TIMEOUT_EPI, &acc_full[b], seg);
                    *abort_flag = 1;
                }
                break;
            }
            tc::tc_fence_after();
            const int n0 = (t / p.m_tiles) * BM, m0 = (t % p.m_tiles) * BN;
            const int row = 32 * q + lane;
            const int n = n0 + row;
            const uint32_t t_acc = tmem + b * BN + ((32u * q) << 16);
            float *slot = p.partials + ((size_t)cta * 2 + (t == first_tile ? 0 : 1)) * (size_t)(BM * BN);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t r[16];
                tc::tmem_ld16(t_acc + c0, r);
                tc::tmem_ld_wait();
                if (whole) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = m0 + c0 + j;
                        if (m < p.M && n < p.N)
                            p.out[(size_t)m * p.N + n] = float_to_bf16_bits(__uint_as_float(r[j]) * __ldg(p.xs + m));
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) slot[(c0 + j) * BM + row] = __uint_as_float(r[j]);
                }
            }
            // release the accumulator buffer to the MMA issuer
            tc::tc_fence_before();
            tc::named_bar_sync(1, 128);
            if (threadIdx.x == EPI_WARP0 * 32) tc::mbar_arrive(&acc_empty[b]);
            if (!whole) {
                // stream-K fix-up: the last contributor of tile t adds the partials in CTA order
                const int c_first = unit_owner(t_lo, p.TU, p.G);
                const int c_last = unit_owner(t_hi - 1, p.TU, p.G);
                __threadfence();
                tc::named_bar_sync(1, 128);
                if (threadIdx.x == EPI_WARP0 * 32) {
                    const int old = atomicAdd(p.counters + t, 1);
                    *last_flag = (old == c_last - c_first);
                }
                tc::named_bar_sync(1, 128);
                if (*last_flag) {
                    __threadfence();
                    // 16 columns at a time, up to 4 contributors' loads in flight together; the
                    // additions still run in CTA order, so the result does not depend on timing
                    const int m_cnt = min(BN, p.M - m0);
                    for (int c0 = 0; c0 < m_cnt; c0 += 16) {
                        float acc[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
                        for (int cb = c_first; cb <= c_last; cb += 4) {
                            float v[4][16];
#pragma unroll
                            for (int cc = 0; cc < 4; ++cc) {
                                const int c = cb + cc;
                                if (c <= c_last) {
                                    const int sl = (t == (int)(unit_start(c, p.TU, p.G) / p.U)) ? 0 : 1;
                                    const float *src = p.partials + ((size_t)c * 2 + sl) * (size_t)(BM * BN) + c0 * BM + row;
#pragma unroll
                                    for (int j = 0; j < 16; ++j) v[cc][j] = __ldcg(src + j * BM);
                                }
                            }
#pragma unroll
                            for (int cc = 0; cc < 4; ++cc)
                                if (cb + cc <= c_last) {
#pragma unroll
                                    for (int j = 0; j < 16; ++j) acc[j] += v[cc][j];
                                }
                        }
                        if (n < p.N) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int m = m0 + c0 + j;
                                if (c0 + j < m_cnt)
                                    p.out[(size_t)m * p.N + n] = float_to_bf16_bits(acc[j] * __ldg(p.xs + m));
                            }
                        }
                    }
                    if (threadIdx.x == EPI_WARP0 * 32) p.counters[t] = 0;
                }
                tc::named_bar_sync(1, 128);  // last_flag is reused by the next tile
            }
            ++seg;
            u = ue;
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        int zero = 0;
        if (*abort_flag) {
            // drain: TMA copies issued but not consumed
            for (int i = *consumed; i < *issued; ++i)
                if (tc::mbar_wait(&full[i % STAGES], (i / STAGES) & 1, &zero, DRAIN_BUDGET)) break;
            for (int g = max(0, *sfr_issued - L::SFR_SLOTS); g < *sfr_issued; ++g)
                tc::mbar_wait(&sfr_full[g % L::SFR_SLOTS], (g / L::SFR_SLOTS) & 1, &zero, DRAIN_BUDGET);
        }
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
    int BN, m_tiles, n_tiles, U, G;
    long long TU;
};

Cfg choose(int64_t M, int64_t N, int64_t K)
{
    Cfg c;
    c.BN = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
    c.n_tiles = (int)((N + BM - 1) / BM);
    c.m_tiles = (int)((M + c.BN - 1) / c.BN);
    c.U = (int)(K / 512);
    c.TU = (long long)c.n_tiles * c.m_tiles * c.U;
    c.G = (int)std::min<long long>(tch::num_sms(), c.TU);
    return c;
}

size_t partial_bytes(const Cfg &c)
{
    size_t b = (size_t)c.G * 2 * BM * c.BN * 4;
    return (b + 255) / 256 * 256;
}

size_t workspace_for(const Cfg &c)
{
    return partial_bytes(c) + (size_t)c.m_tiles * c.n_tiles * 4;
}

template <int BN, int STAGES, int PSTAGES, int ACC_BUFS, bool CONV>
w4a8_status launch(const uint8_t *wp, const uint8_t *xq, const Params &prm, cudaStream_t stream)
{
    using L = Layout<BN, STAGES, PSTAGES, ACC_BUFS, CONV>;
    CUtensorMap tw, tx, tsf;
    const bool wmap = CONV ? tch::tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, wp, prm.N, prm.K / 2, prm.K / 2, BM,
                                          64, CU_TENSOR_MAP_SWIZZLE_NONE)
                           : tch::tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, wp, prm.N, prm.K, prm.K / 2,
                                          BM, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!wmap ||
        !tch::tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, prm.M, prm.K, prm.K, BN, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tch::tmap_2d(&tsf, CU_TENSOR_MAP_DATA_TYPE_UINT8, prm.we, prm.N, prm.K / 32, prm.K / 32, BM, 16,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
        return W4A8_ERR_CUDA;
    auto kern = mxfp4_tc_kernel<BN, STAGES, PSTAGES, ACC_BUFS, CONV>;
    static int attr_done[64] = {0};
    if (!tch::set_smem_once(kern, L::TOTAL, attr_done)) return W4A8_ERR_CUDA;
    kern<<<prm.G, NUM_THREADS, L::TOTAL, stream>>>(tw, tx, tsf, prm);
    return w4a8_launch_status();
}

}  // namespace tcg
}  // namespace w4a8

using namespace w4a8::tcg;

bool w4a8_tc_mxfp4_supported(const void *xq, const void *wp, const void *we, const void *out, int64_t M,
                             int64_t N, int64_t K)
{
    // TMA needs 16-byte-strided scale rows (K a multiple of 512), a 32-byte aligned 4-bit tensor
    // and 16-byte aligned byte tensors.
    if (K % 512 != 0 || K > (1ll << 30) || M < 1 || M > (1ll << 30) || N < 1 || N > (1ll << 30))
        return false;
    if (!w4a8_aligned(wp, 32) || !w4a8_aligned(xq, 16) || !w4a8_aligned(we, 16) || !w4a8_aligned(out, 2))
        return false;
    return w4a8::tch::encode_fn() != nullptr;
}

size_t w4a8_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, int policy)
{
    if (policy == 1 || K % 512 != 0 || K <= 0 || M <= 0 || N <= 0) return 0;
    return workspace_for(choose(M, N, K));
}

w4a8_status w4a8_launch_mxfp4_tc(const uint8_t *xq, const float *x_scale, const uint8_t *wp, const uint8_t *we,
                                 uint16_t *out, int64_t M, int64_t N, int64_t K, void *workspace, int,
                                 cudaStream_t stream)
{
    const Cfg c = choose(M, N, K);
    Params prm;
    prm.we = we;
    prm.xs = x_scale;
    prm.out = out;
    prm.partials = static_cast<float *>(workspace);
    prm.counters = reinterpret_cast<int *>(static_cast<uint8_t *>(workspace) + partial_bytes(c));
    prm.status = w4a8_device_status_ptr();
    if (!prm.status) return W4A8_ERR_CUDA;
    prm.M = (int)M;
    prm.N = (int)N;
    prm.K = (int)K;
    prm.m_tiles = c.m_tiles;
    prm.n_tiles = c.n_tiles;
    prm.U = c.U;
    prm.TU = c.TU;
    prm.G = c.G;
    prm.trace = static_cast<unsigned long long *>(w4a8_debug_trace_ptr());
    if (w4a8_gemm_policy() == 3) {  // converter variant (diagnostics)
        switch (c.BN) {
        case 16: return launch<16, 12, 3, 2, true>(wp, xq, prm, stream);
        case 32: return launch<32, 12, 3, 2, true>(wp, xq, prm, stream);
        case 64: return launch<64, 10, 3, 2, true>(wp, xq, prm, stream);
        case 128: return launch<128, 6, 3, 2, true>(wp, xq, prm, stream);
        default: return launch<256, 4, 2, 1, true>(wp, xq, prm, stream);
        }
    }
    switch (c.BN) {
    case 16: return launch<16, 12, 1, 2, false>(wp, xq, prm, stream);
    case 32: return launch<32, 10, 1, 2, false>(wp, xq, prm, stream);
    case 64: return launch<64, 8, 1, 2, false>(wp, xq, prm, stream);
    case 128: return launch<128, 6, 1, 2, false>(wp, xq, prm, stream);
    default: return launch<256, 4, 1, 1, false>(wp, xq, prm, stream);
    }
}

// int4 tensor-core path: not yet; every int4 call takes the CUDA-core kernel.
bool w4a8_tc_int4_supported(const void *, const void *, const void *, const void *, int64_t, int64_t, int64_t)
{
    return false;
}
size_t w4a8_tc_int4_workspace_bytes(int64_t, int64_t, int64_t, int) { return 0; }
w4a8_status w4a8_launch_int4_tc(const uint8_t *, const float *, const int32_t *, const uint16_t *, uint16_t *,
                                int64_t, int64_t, int64_t, void *, int, cudaStream_t)
{
    return W4A8_ERR_UNSUPPORTED_SHAPE;
}
