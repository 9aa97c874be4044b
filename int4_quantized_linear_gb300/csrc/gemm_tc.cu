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
//   * TMA: one 3-D box brings KPU consecutive k-tiles (128 K each) of 128 weight rows, already in
//     the padded form the instruction reads for 4-bit operands (16U4_ALIGN16B: 16 codes in the
//     low 8 bytes of each 16-byte slot) with the 128-byte swizzle; another brings the matching
//     activation tiles; the weight scales come as one [128 rows x 16 bytes] tile per 4 k-tiles.
//     Boxes whose rows read 4 k-tiles (256 contiguous bytes) at once run TMA at the full HBM
//     rate on GB300, where one-k-tile boxes (64-byte rows) reach only about 60% of it;
//   * four scale warps (one per TMEM lane quarter) write each row's 4-byte scale word, repeated
//     over 4 columns, into tensor memory with tcgen05.st; the MMA reads one byte per k-block;
//   * persistent stream-K: one CTA per SM walks a contiguous range of (tile, 4-k-tile unit)
//     work, so the TMA ring never drains between tiles and every SM gets the same number of
//     units; a tile whose K range is split between CTAs is finished by the last contributor,
//     which adds the fp32 partials in CTA order;
//   * two accumulator buffers in tensor memory (one for 256-token tiles) let the MMAs of the next
//     tile run while the epilogue drains the previous one;
//   * the MMA-issuing thread never touches shared memory inside its loop: on GB300 any shared-memory
//     access by a thread with MMAs in flight (an mbarrier test included) waits for those MMAs to
//     complete, which drains the tensor pipe every k-tile.  A gate warp does all the mbarrier
//     waiting and releases the MMA warp one k-tile at a time through a hardware named barrier;
//   * warp roles: 0 TMA producer, 1 TMEM allocator + MMA issuer, 2-5 scale warps, 6-9 epilogue,
//     10 gate (scale and epilogue warps each use the TMEM lane quarter their warp index selects).
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
constexpr int NUM_THREADS = 352;   // 11 warps
constexpr int SCALE_WARP0 = 2;     // warps 2-5
constexpr int EPI_WARP0 = 6;       // warps 6-9
constexpr int GATE_WARP = 10;
constexpr int GATE_BARRIER = 2;    // named barrier shared by the gate warp and the MMA warp
constexpr long long WAIT_BUDGET = 1ll << 29;  // clock cycles (a quarter second or so)
constexpr long long DRAIN_BUDGET = 1ll << 24;

enum : unsigned { ST_TIMEOUT_PRODUCER = 1, ST_TIMEOUT_GATE = 2, ST_TIMEOUT_SCALE = 4, ST_TIMEOUT_EPI = 8 };

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
enum { TR_TMA_ISSUED = 0, TR_SCALE_DATA, TR_SCALE_DONE, TR_MMA_READY, TR_MMA_ISSUED, TR_UNUSED, TR_EVENTS };
__device__ __forceinline__ void trace_ev(const Params &p, int ev, int i)
{
    if (p.trace != nullptr && blockIdx.x == 0 && i < TRACE_N) p.trace[ev * TRACE_N + i] = (unsigned long long)clock64();
}
// Phase stamps (global timer, ns) of every CTA (up to 512): entry, set-up done, epilogue done,
// exit (k = 0..3), and for the last tile the epilogue's accumulator ready, partial stored,
// arrival counted, fix-up done (k = 4..7); at [TR_EVENTS * TRACE_N + 8 * cta + k].
__device__ __forceinline__ void trace_phase(const Params &p, int k)
{
    if (p.trace != nullptr && blockIdx.x < 512) {
        unsigned long long ns;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ns));
        p.trace[TR_EVENTS * TRACE_N + 8 * blockIdx.x + k] = ns;
    }
}

// Shared memory: a ring of US slots, each holding KPU k-tiles of padded weights (16 KB each)
// and activations (BN x 128 bytes each), plus a ring of 2 raw scale tiles (4 k-tiles each).
template <int BN, int KPU, int US, int ACC_BUFS>
struct Layout {
    static constexpr int W_TILE = BM * 128;             // one padded weight k-tile
    static constexpr int X_TILE = BN * 128;             // one activation k-tile (swizzled)
    static constexpr int W_SLOT = KPU * W_TILE;
    static constexpr int X_SLOT = KPU * X_TILE;
    static constexpr int SFR_SLOTS = 2;
    static constexpr int SFR_BYTES = BM * 16;
    static constexpr int W_OFF = 0;
    static constexpr int X_OFF = W_OFF + US * W_SLOT;
    static constexpr int SFR_OFF = X_OFF + US * X_SLOT;
    static constexpr int BAR_OFF = SFR_OFF + SFR_SLOTS * SFR_BYTES;
    static constexpr int TOTAL = BAR_OFF + 1024 + 1024;  // barriers, flags, alignment slack
    static constexpr int TX_BYTES = KPU * (BM * 64 + X_TILE);  // 4-bit boxes count packed bytes
    static constexpr int SF_SLOTS = KPU * US;           // TMEM scale slots, 4 columns each
    static constexpr int T_SFB = ACC_BUFS * BN;         // TMEM column of the unit B scales
    static constexpr int T_SFA = T_SFB + 8;             // TMEM columns of the A scales
    static constexpr int TMEM_NEED = T_SFA + 4 * SF_SLOTS;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64
                                     : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
    static_assert(4 % KPU == 0, "a ring slot lies inside one 4-k-tile unit");
    static_assert(TMEM_NEED <= 512, "tensor memory");
    static_assert(TOTAL <= 232448, "shared memory");
    static_assert((X_TILE % 1024) == 0 && (X_OFF % 1024) == 0, "swizzled tiles are 1024-aligned");
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

// Bounded wait by one thread that records a timeout and raises the abort flag; 0 = done.
__device__ __forceinline__ int wait_or_fail(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                            unsigned int *status, unsigned int bit, int iter)
{
    const int w = tc::mbar_wait(bar, parity, abort_flag, WAIT_BUDGET);
    if (w == 1) fail(status, bit, bar, iter);
    if (w) *abort_flag = 1;
    return w;
}

// Warp-uniform version: lane 0 waits, the result is broadcast.
__device__ __forceinline__ int warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         unsigned int *status, unsigned int bit, int iter, int lane)
{
    int w = 0;
    if (lane == 0) w = wait_or_fail(bar, parity, abort_flag, status, bit, iter);
    return __shfl_sync(0xffffffffu, w, 0);
}

template <int BN, int KPU, int US, int ACC_BUFS>
__global__ void __launch_bounds__(NUM_THREADS, 1)
mxfp4_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_sf, const Params p)
{
    using L = Layout<BN, KPU, US, ACC_BUFS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);  // ring slot landed
    uint64_t *empty = full + US;                                        // ring slot free again
    uint64_t *sff = empty + US;                                         // fill's scales in TMEM
    uint64_t *sfr_full = sff + US;
    uint64_t *sfr_empty = sfr_full + L::SFR_SLOTS;
    uint64_t *acc_full = sfr_empty + L::SFR_SLOTS;
    uint64_t *acc_empty = acc_full + ACC_BUFS;
    uint64_t *mma_done = acc_empty + ACC_BUFS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *last_flag = reinterpret_cast<int *>(tmem_slot + 2);
    int *issued = reinterpret_cast<int *>(tmem_slot + 4);     // ring fills issued
    int *sfr_issued = reinterpret_cast<int *>(tmem_slot + 5);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u_begin = unit_start(cta, p.TU, p.G);
    const long long u_end = unit_start(cta + 1, p.TU, p.G);
    const int n_k = (int)(4 * (u_end - u_begin));  // k-tiles this CTA processes
    if (threadIdx.x == 0) trace_phase(p, 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < US; ++s) {
            tc::mbar_init(&full[s], 1);   // producer expect_tx
            tc::mbar_init(&empty[s], 1);  // tcgen05.commit after the slot's last MMAs
        }
        for (int s = 0; s < US; ++s) tc::mbar_init(&sff[s], 4);  // one arrival per scale warp
        for (int r = 0; r < L::SFR_SLOTS; ++r) {
            tc::mbar_init(&sfr_full[r], 1);
            tc::mbar_init(&sfr_empty[r], 4);
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            tc::mbar_init(&acc_full[b], 1);   // tcgen05.commit after a tile's last MMA
            tc::mbar_init(&acc_empty[b], 1);  // epilogue finished reading the buffer
        }
        tc::mbar_init(mma_done, 1);
        *abort_flag = 0;
        *last_flag = 0;
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
    if (threadIdx.x == 0) trace_phase(p, 1);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int i = 0; i < n_k && !*abort_flag; i += KPU) {
                const long long u = u_begin + i / 4;
                const int t = (int)(u / p.U);
                const int kt = (int)(u - (long long)t * p.U) * 4 + (i & 3);  // first k-tile of the fill
                const int n0 = (t / p.m_tiles) * BM, m0 = (t % p.m_tiles) * BN;
                if ((i & 3) == 0) {
                    const int g = i >> 2, rs = g % L::SFR_SLOTS;
                    if (wait_or_fail(&sfr_empty[rs], ((g / L::SFR_SLOTS) & 1) ^ 1, abort_flag, p.status,
                                     ST_TIMEOUT_PRODUCER, g))
                        break;
                    tc::mbar_arrive_expect_tx(&sfr_full[rs], L::SFR_BYTES);
                    tc::tma_load_2d(smem + L::SFR_OFF + rs * L::SFR_BYTES, &tmap_sf, &sfr_full[rs], 4 * kt, n0);
                    *sfr_issued = g + 1;
                }
                const int f = i / KPU, sl = f % US;
                if (wait_or_fail(&empty[sl], ((f / US) & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER, i))
                    break;
                tc::mbar_arrive_expect_tx(&full[sl], L::TX_BYTES);
                tc::tma_load_3d(smem + L::W_OFF + sl * L::W_SLOT, &tmap_w, &full[sl], 0, n0, kt);
                tc::tma_load_3d(smem + L::X_OFF + sl * L::X_SLOT, &tmap_x, &full[sl], 0, m0, kt);
                *issued = f + 1;
                trace_ev(p, TR_TMA_ISSUED, i);
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == GATE_WARP) {
        // ------------------------------------------------------------ MMA issuer and its gate
        // Both warps walk the same sequence of ring fills (KPU k-tiles each) and meet at the named
        // barrier once per fill (also after an abort, so neither can be left waiting there).  The
        // gate first waits for the fill's scales -- written after its data landed -- and, at the
        // first fill of a tile, for the accumulator buffer; the MMA warp then issues the fill's
        // 4 x KPU MMAs without touching memory.
        const bool gate = (warp == GATE_WARP);
        if (!gate) tc::tc_fence_after();
        int f = 0, seg = 0;
        long long u = u_begin;
        while (u < u_end) {
            const int t = (int)(u / p.U);
            const long long ue = min(u_end, (long long)(t + 1) * p.U);
            const int b = seg % ACC_BUFS;
            const uint32_t t_acc = tmem + b * BN;
            const int f_end = f + (int)(4 * (ue - u)) / KPU;
            for (bool first = true; f < f_end; ++f, first = false) {
                const int sl = f % US;
                if (gate) {
                    if (!*abort_flag && first)
                        warp_wait(&acc_empty[b], ((seg / ACC_BUFS) & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_GATE, seg, lane);
                    if (!*abort_flag)
                        warp_wait(&sff[sl], (f / US) & 1, abort_flag, p.status, ST_TIMEOUT_GATE, f, lane);
                    if (lane == 0) trace_ev(p, TR_MMA_READY, f);
                }
                // the gate's abort state rides on the barrier: the MMA thread reads no memory here
                const bool aborted = tc::named_bar_or(GATE_BARRIER, 64, gate && *abort_flag);
                if (!gate && lane == 0 && !aborted) {
                    tc::tc_fence_after();
#pragma unroll
                    for (int j = 0; j < KPU; ++j) {
                        const uint32_t sfa = tmem + L::T_SFA + 4 * (sl * KPU + j);
                        const uint32_t wa = tc::smem_u32(smem + L::W_OFF + sl * L::W_SLOT + j * L::W_TILE);
                        const uint32_t xa = tc::smem_u32(smem + L::X_OFF + sl * L::X_SLOT + j * L::X_TILE);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = tc::smem_desc(wa + 32 * kk, 16, 1024, 2);
                            const uint64_t bd = tc::smem_desc(xa + 32 * kk, 16, 1024, 2);
                            tc::mma_mxf8f6f4(t_acc, ad, bd, tc::idesc_mxf8f6f4(5, 0, BM, BN, kk, 0), sfa,
                                             tmem + L::T_SFB, (first && j == 0 && kk == 0) ? 0u : 1u);
                        }
                    }
                    tc::tc_commit(&empty[sl]);
                    if (f_end - f == 1) tc::tc_commit(&acc_full[b]);
                }
                __syncwarp();
            }
            ++seg;
            u = ue;
        }
        if (!gate && lane == 0) tc::tc_commit(mma_done);  // teardown waits on it before freeing TMEM
        __syncwarp();
    } else if (warp < EPI_WARP0) {
        // ------------------------------------------------------------ scale warps (2-5)
        // Warp w owns TMEM lanes 32q..32q+31, q = w & 3 (weight rows 32q..32q+31).  For each
        // k-tile of a ring fill it writes its rows' 4-byte scale word (the 4 k-block scales of
        // that k-tile) into the 4 columns of the fill's TMEM scale slot.  Those columns were last
        // read by the MMAs of the previous fill of the same ring slot; the producer refilled the
        // ring slot only after those MMAs finished, so waiting for the fill covers it.
        const int q = warp & 3;
        const int row = 32 * q + lane;
        int w = 0;
        for (int i = 0; i < n_k && !w; i += KPU) {
            const int g = i >> 2, rs = g % L::SFR_SLOTS;
            if ((i & 3) == 0 &&
                (w = warp_wait(&sfr_full[rs], (g / L::SFR_SLOTS) & 1, abort_flag, p.status, ST_TIMEOUT_SCALE, g, lane)))
                break;
            const int f = i / KPU, sl = f % US;
            if ((w = warp_wait(&full[sl], (f / US) & 1, abort_flag, p.status, ST_TIMEOUT_SCALE, f, lane)))
                break;
            if (lane == 0 && warp == SCALE_WARP0) trace_ev(p, TR_SCALE_DATA, f);
            const uint8_t *raw = smem + L::SFR_OFF + rs * L::SFR_BYTES + row * 16;
#pragma unroll
            for (int j = 0; j < KPU; ++j) {
                const uint32_t sw = *reinterpret_cast<const uint32_t *>(raw + 4 * ((i & 3) + j));
                tc::tmem_st4(tmem + L::T_SFA + 4 * (sl * KPU + j) + ((32u * q) << 16), sw, sw, sw, sw);
            }
            tc::tmem_st_wait();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&sff[sl]);
                if (((i + KPU) & 3) == 0) tc::mbar_arrive(&sfr_empty[rs]);
                if (warp == SCALE_WARP0) trace_ev(p, TR_SCALE_DONE, f);
            }
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
            const bool last_seg = (ue == u_end);
            if (last_seg && threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 4);
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
                if (last_seg && threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 5);
                __threadfence();
                tc::named_bar_sync(1, 128);
                if (threadIdx.x == EPI_WARP0 * 32) {
                    const int old = atomicAdd(p.counters + t, 1);
                    *last_flag = (old == c_last - c_first);
                }
                tc::named_bar_sync(1, 128);
                if (last_seg && threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 6);
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
                if (last_seg && threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 7);
            }
            ++seg;
            u = ue;
        }
        if (threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 2);
    }


    tc::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        int zero = 0;
        if (*abort_flag) {
            // drain: TMA copies issued but not waited for
            for (int f = max(0, *issued - US); f < *issued; ++f)
                if (tc::mbar_wait(&full[f % US], (f / US) & 1, &zero, DRAIN_BUDGET)) break;
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
    if (threadIdx.x == 0) trace_phase(p, 3);
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

template <int BN, int KPU, int US, int ACC_BUFS>
w4a8_status launch(const uint8_t *wp, const uint8_t *xq, const Params &prm, cudaStream_t stream)
{
    using L = Layout<BN, KPU, US, ACC_BUFS>;
    CUtensorMap tw, tx, tsf;
    // 3-D views [k-tile][row][128 K]: weights (4-bit codes; a row is K/2 bytes, a k-tile 64) and
    // activations (bytes; a row is K bytes, a k-tile 128)
    if (!tch::tmap_3d_ktiles(&tw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, wp, prm.N, prm.K / 2, 64, prm.K / 128, BM,
                             KPU) ||
        !tch::tmap_3d_ktiles(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, prm.M, prm.K, 128, prm.K / 128, BN, KPU) ||
        !tch::tmap_2d(&tsf, CU_TENSOR_MAP_DATA_TYPE_UINT8, prm.we, prm.N, prm.K / 32, prm.K / 32, BM, 16,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
        return W4A8_ERR_CUDA;
    auto kern = mxfp4_tc_kernel<BN, KPU, US, ACC_BUFS>;
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

size_t w4a8_tc_workspace_counters_offset(int64_t M, int64_t N, int64_t K)
{
    return partial_bytes(choose(M, N, K));
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
    switch (c.BN) {
    case 16: return launch<16, 4, 3, 2>(wp, xq, prm, stream);
    case 32: return launch<32, 4, 2, 2>(wp, xq, prm, stream);
    case 64: return launch<64, 4, 2, 2>(wp, xq, prm, stream);
    case 128: return launch<128, 2, 3, 2>(wp, xq, prm, stream);
    default: return launch<256, 2, 2, 1>(wp, xq, prm, stream);
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
