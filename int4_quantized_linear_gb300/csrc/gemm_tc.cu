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
//     over 4 columns, into a ring of tensor-memory scale slots with tcgen05.st; the MMA reads one
//     byte per k-block.  The raw scale tiles are loaded a few units ahead of the data (the first
//     ones by the producer, each later one by a scale warp as soon as the tile it replaces has been
//     read, so a scale load never holds up a data load) and a TMEM slot only waits for the MMAs
//     that last read it, so scale work stays off the TMA -> MMA path;
//   * persistent stream-K: one CTA per SM walks a contiguous range of (tile, 4-k-tile unit)
//     work, so the TMA ring never drains between tiles and every SM gets the same number of
//     units; a tile whose K range is split between CTAs is finished by the last contributor,
//     which adds the fp32 partials in CTA order.  Each CTA takes its split tiles first, so their
//     fix-up overlaps the whole tiles' MMAs; at the CTA's last tile the ring is idle, and bulk
//     copies bring every contributor's partial into it in one round trip;
//   * two accumulator buffers in tensor memory (one for 256-token tiles) let the MMAs of the next
//     tile run while the epilogue drains the previous one; output leaves through a small shared
//     memory staging buffer and TMA tensor stores (per-thread 2-byte stores ran at a fraction of
//     that rate with most of the L1/shared array given to shared memory);
//   * the MMA-issuing thread never touches shared memory inside its loop: on GB300 any shared-memory
//     access by a thread with MMAs in flight (an mbarrier test included) waits for those MMAs to
//     complete, which drains the tensor pipe every k-tile.  A gate warp does all the mbarrier
//     waiting and releases the MMA warp one ring fill at a time through a hardware named barrier;
//   * programmatic dependent launch: barrier set-up and tensor-memory allocation overlap the
//     previous kernel in the stream; inputs and outputs are touched only after griddepcontrol.wait;
//   * warp roles: 0 TMA producer, 1 TMEM allocator + MMA issuer, 2-5 scale warps, 6-9 epilogue,
//     10 gate (scale and epilogue warps each use the TMEM lane quarter their warp index selects).
//
// W4A4 ("vllm-radiance (MXFP4)", section "Native MXFP4": MXFP4 activations too, group 32, e8m0):
// the A4 instantiations read the activations as 4-bit codes through the same padded TMA form
// as the weights and give the instruction both operands as e2m1 (the same kind::mxf8f6f4
// instruction, B format e2m1).  The activation scales come as [BN tokens x 16 bytes] tiles
// beside each weight scale tile and the scale warps write them into a ring of B-scale slots:
// token t's 4-byte word (its 4 k-block scales of a k-tile) in lane t % 32 of every lane
// quarter, column t / 32 of the slot.  There is no per-token scale.
//
// Every mbarrier wait is bounded; a wait that runs out sets a bit in the library's device status
// word and the CTA winds down (draining what it started) instead of hanging.
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "dispatch.h"
#include "tc_host.cuh"
#include "tc_ptx.cuh"
#include "tc_sched.cuh"

namespace w4a8 {
namespace tcg {

using namespace tcs;

constexpr int NUM_THREADS = 352;   // 11 warps
// With the activation quant fused in (AQ) the four scale warps also write each ring fill's
// activation codes: no extra warps, so the kernel keeps 168 registers per thread (more warps would
// cut that to 128 and spill; with shared memory taking nearly all of the L1 array, every spill
// reload is an L2 round trip).
constexpr int AQ_BARRIER = 3;         // named barrier of the row-amax step (scale + epilogue warps)
constexpr int AQ_STEP_THREADS = 256;
constexpr int SCALE_WARP0 = 2;     // warps 2-5
constexpr int EPI_WARP0 = 6;       // warps 6-9
constexpr int GATE_WARP = 10;
constexpr int GATE_BARRIER = 2;    // named barrier shared by the gate warp and the MMA warp

enum : unsigned { ST_TIMEOUT_PRODUCER = 1, ST_TIMEOUT_GATE = 2, ST_TIMEOUT_SCALE = 4, ST_TIMEOUT_EPI = 8,
                  ST_TIMEOUT_AQ = 16 };
constexpr int AQ_MAX_M = 2;        // tokens the fused activation quant takes (4 values per token and scale-warp thread)

struct Params {
    const uint8_t *wp;     // [N, K/2] packed e2m1 codes
    const uint8_t *we;     // [N, K/32] e8m0
    const float *xs;       // [M] per-token scale
    const uint16_t *x;     // AQ: [M, K] bf16 activations, quantized inside the kernel
    uint16_t *out;         // [M, N] bf16
    float *partials;       // [G][2][BN][128] fp32 stream-K partial tiles
    int *counters;         // arrival counters of the split tiles (index < G), zero between calls
    unsigned int *status;  // device status block
    int M, N, K;
    int m_tiles, n_tiles;
    int U;                 // 4-k-tile units per tile
    long long RU;          // stream-K units (those of the first R tiles)
    int R, D;              // stream-K tiles; whole tiles per CTA after them
    int G, Gsk;            // CTAs; CTAs sharing the stream-K units
    int evict_first;       // weights are read once: load them with the L2 evict-first policy
    int tma_out;           // output tiles leave through shared memory and TMA stores (else plain stores)
    int w_early;           // the first ring fills' weights and scales may be loaded before the
                           // wait on the previous kernel (it is known not to write them)
    unsigned long long *trace;  // optional pipeline timeline of CTA 0 (diagnostics), or null
};

// Pipeline timeline (a development aid, compiled in only when W4A8_TRACE is defined): CTA 0
// records clock64() per k-tile i < TRACE_N for each event.
constexpr int TRACE_N = 256;
enum { TR_TMA_ISSUED = 0, TR_SCALE_DATA, TR_SCALE_DONE, TR_MMA_READY, TR_TMA_FILL, TR_GATE_SFF, TR_AQ_SLOT, TR_AQ_DONE,
       TR_EVENTS };
__device__ __forceinline__ void trace_ev(const Params &p, int ev, int i)
{
#ifdef W4A8_TRACE
    if (p.trace != nullptr && blockIdx.x == 0 && i < TRACE_N) p.trace[ev * TRACE_N + i] = (unsigned long long)clock64();
#endif
}
// Phase stamps (global timer, ns) of every CTA (up to 512), at [TR_EVENTS * TRACE_N + 16 * cta + k]:
// k = 0 entry, 1 set-up done, 2 epilogue done, 3 exit; for the CTA's last tile the epilogue's
// 4 accumulator ready, 5 partial stored, 6 arrival counted, 7 fix-up done; 8 first fill released
// to the MMA warp, 9 last fill released, 10 MMA warp done issuing, 11 first accumulator ready,
// 12 last tile's partials staged in shared memory, 13 summed and stored, 14 / 15 its first 16
// columns summed / stored.
constexpr int TRACE_PHASES = 16;
__device__ __forceinline__ void trace_phase(const Params &p, int k)
{
#ifdef W4A8_TRACE
    if (p.trace != nullptr && blockIdx.x < 512) {
        unsigned long long ns;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ns));
        p.trace[TR_EVENTS * TRACE_N + TRACE_PHASES * blockIdx.x + k] = ns;
    }
#endif
}

// Fused activation quant, first step, run by the quantizer and epilogue warps together
// (AQ_STEP_THREADS threads, pidx 0 .. AQ_STEP_THREADS - 1): each token row's amax over all K, taken on the bf16 bit patterns (for
// finite values |x| orders like the 15 low bits) as w4a8_act_quant takes it, then the per-token
// scale amax / 448 (correctly rounded; 1.0 for an all-zero row) into s_out[m].  The rows are read
// from L2 in batches of BATCH 16-byte chunks per thread, so each thread keeps that many loads in
// flight (every thread walks the same chunks whatever its batch size).
template <int BATCH>
__device__ __forceinline__ void aq_row_scales(const uint16_t *x, int M, int K, int pidx, float *s_out, unsigned *rmax)
{
    if (pidx < M) rmax[pidx] = 0u;
    tc::named_bar_sync(AQ_BARRIER, AQ_STEP_THREADS);
    const int nchunk = K / 8;
    const int total = M * nchunk;
    const uint4 *src = reinterpret_cast<const uint4 *>(x);
    int m_cur = pidx / nchunk;
    uint32_t a2 = 0;  // two 15-bit magnitudes packed, per-halfword max
    auto flush = [&]() {
        const uint32_t hb = max(a2 & 0xffffu, a2 >> 16);
        if (hb) atomicMax(&rmax[m_cur], hb);
    };
    for (int base = pidx; base < total; base += BATCH * AQ_STEP_THREADS) {
        uint4 v[BATCH];
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            const int idx = base + j * AQ_STEP_THREADS;
            v[j] = idx < total ? __ldg(src + idx) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            const int idx = base + j * AQ_STEP_THREADS;
            if (idx < total) {
                const int m = idx / nchunk;
                if (m != m_cur) {
                    flush();
                    m_cur = m;
                    a2 = 0;
                }
                a2 = __vmaxu2(a2, v[j].x & 0x7fff7fffu);
                a2 = __vmaxu2(a2, v[j].y & 0x7fff7fffu);
                a2 = __vmaxu2(a2, v[j].z & 0x7fff7fffu);
                a2 = __vmaxu2(a2, v[j].w & 0x7fff7fffu);
            }
        }
    }
    if (pidx < total) flush();
    tc::named_bar_sync(AQ_BARRIER, AQ_STEP_THREADS);
    if (pidx < M) {
        const float amax = bf16_bits_to_float(rmax[pidx]);
        s_out[pidx] = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    }
    tc::named_bar_sync(AQ_BARRIER, AQ_STEP_THREADS);
}

// Shared memory: a ring of US slots, each holding KPU k-tiles of padded weights (16 KB each)
// and activations (BN x 128 bytes each), plus a ring of SFR raw scale tiles (4 k-tiles each).
// Tensor memory: ACC_BUFS accumulators of BN columns, the unit B scales, and a ring of SFQ
// scale slots (KPU k-tiles of A scales each) that the scale warps fill ahead of the data.  With
// SFQ == US (the decode tilings) a scale slot is tied to its ring slot and freed by the same
// commit, one commit per fill fewer.
template <int BN, int KPU, int US, int ACC_BUFS, int SFQ, int SFR, bool A4 = false, bool AQ = false>
struct Layout {
    static constexpr int W_TILE = BM * 128;             // one padded weight k-tile
    static constexpr int X_TILE = BN * 128;             // one activation k-tile (swizzled)
    static constexpr int W_SLOT = KPU * W_TILE;
    static constexpr int X_SLOT = KPU * X_TILE;
    static constexpr int SFR_SLOTS = SFR;
    static constexpr int SFR_BYTES = BM * 16 + (A4 ? BN * 16 : 0);  // weight (+ activation) scale tiles
    static constexpr int SFR_B_OFF = BM * 16;           // the activation scale tile in a raw slot
    static constexpr int W_OFF = 0;
    static constexpr int X_OFF = W_OFF + US * W_SLOT;
    static constexpr int SFR_OFF = X_OFF + US * X_SLOT;
    static constexpr int BAR_OFF = SFR_OFF + SFR_SLOTS * SFR_BYTES;
    static constexpr int XS_OFF = BAR_OFF + 512;        // barriers and flags below, then the tile's token scales
    static constexpr int NSTAGE = BN == 16 ? 1 : 2;     // output staging: [16 tokens][128 rows] bf16 buffers
    static constexpr int STAGE_BYTES = 16 * BM * 2;
    static constexpr int AQ_OFF = XS_OFF + BN * 4;      // AQ: per-token scales [BN], row maxima [BN]
    static constexpr int AQ_BYTES = AQ ? 2 * BN * 4 : 0;
    static constexpr int STAGE_OFF = (AQ_OFF + AQ_BYTES + 1023) / 1024 * 1024;
    static constexpr int TOTAL = STAGE_OFF + NSTAGE * STAGE_BYTES + 1024;  // + alignment slack
    static constexpr int TX_BYTES = KPU * (BM * 64 + (A4 ? BN * 64 : AQ ? 0 : X_TILE));  // 4-bit boxes count packed bytes
    static constexpr int SF_SLOTS = KPU * SFQ;          // TMEM scale k-tile slots, 4 columns each
    static constexpr int SFBW = BN <= 128 ? 4 : 8;      // W4A4: TMEM columns per B-scale k-tile slot
    static constexpr int T_SFB = ACC_BUFS * BN;         // TMEM column of the B scales (unit, or W4A4's ring)
    static constexpr int T_SFA = T_SFB + (A4 ? SFBW * SF_SLOTS : 8);  // TMEM columns of the A scales
    static constexpr int TMEM_NEED = T_SFA + 4 * SF_SLOTS;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64
                                     : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
    static_assert(4 % KPU == 0, "a ring slot lies inside one 4-k-tile unit");
    static_assert(TMEM_NEED <= 512, "tensor memory");
    static_assert(TOTAL <= 232448, "shared memory");
    static_assert(8 * (2 * US + 2 * SFQ + 2 * SFR + 2 * ACC_BUFS + 2) + 32 <= 512, "barrier area");
    static_assert((X_TILE % 1024) == 0 && (X_OFF % 1024) == 0, "swizzled tiles are 1024-aligned");
};

// Stream-K fix-up of a decode tile (up to 64 tokens): whole partials of a group of contributors
// per round trip to L2 pays when that takes fewer trips than one per 16-column chunk (64-token
// tiles with at most three contributors; 32-token tiles always, three contributors a trip).
template <int BN>
__device__ __forceinline__ bool narrow_fixup(int n_contrib)
{
    if constexpr (BN > 64) return false;
    else if constexpr (BN == 64) return n_contrib < 4;
    else return BN == 32;  // 16-token tiles: the chunked path below is the same thing
}

template <int BN, int KPU, int US, int ACC_BUFS, int SFQ, int SFR, bool A4, bool AQ>
__global__ void __launch_bounds__(NUM_THREADS, 1)
mxfp4_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_sf, const __grid_constant__ CUtensorMap tmap_out,
                const __grid_constant__ CUtensorMap tmap_sfb, const Params p)
{
    using L = Layout<BN, KPU, US, ACC_BUFS, SFQ, SFR, A4, AQ>;
    static_assert(!(AQ && (A4 || BN != 16)), "the fused activation quant serves the 16-token decode tiling");
    static_assert(!AQ || KPU * 128 / 4 == 128, "one 4-value chunk per token, scale-warp thread and fill");
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived by pointer arithmetic so the compiler keeps it in the shared window
    uint8_t *smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);  // ring slot landed
    uint64_t *empty = full + US;                                        // ring slot free again
    uint64_t *sff = empty + US;                                         // fill's scales in TMEM
    uint64_t *sfe = sff + SFQ;                                          // TMEM scale slot free again
    uint64_t *sfr_full = sfe + SFQ;
    uint64_t *sfr_empty = sfr_full + L::SFR_SLOTS;
    uint64_t *acc_full = sfr_empty + L::SFR_SLOTS;
    uint64_t *acc_empty = acc_full + ACC_BUFS;
    uint64_t *mma_done = acc_empty + ACC_BUFS;
    uint64_t *fix_bar = mma_done + 1;  // partials staged for the last tile's fix-up
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fix_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *last_flag = reinterpret_cast<int *>(tmem_slot + 2);
    int *issued = reinterpret_cast<int *>(tmem_slot + 4);     // ring fills issued
    int *sfr_issued = reinterpret_cast<int *>(tmem_slot + 5);
    int *fix_issued = reinterpret_cast<int *>(tmem_slot + 6);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const Sched sched(cta, p.Gsk, p.RU, p.D, p.R, p.U);
    const int n_k = 4 * sched.n_units;  // k-tiles this CTA processes
    if (threadIdx.x == 0) trace_phase(p, 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < US; ++s) {
            tc::mbar_init(&full[s], AQ ? 5 : 1);  // producer expect_tx (+ the four scale warps)
            tc::mbar_init(&empty[s], 1);  // tcgen05.commit after the slot's last MMAs
        }
        for (int s = 0; s < SFQ; ++s) {
            tc::mbar_init(&sff[s], 4);  // one arrival per scale warp
            tc::mbar_init(&sfe[s], 1);  // tcgen05.commit after the slot's MMAs
        }
        for (int r = 0; r < L::SFR_SLOTS; ++r) {
            tc::mbar_init(&sfr_full[r], 1);
            tc::mbar_init(&sfr_empty[r], 4);
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            tc::mbar_init(&acc_full[b], 1);   // tcgen05.commit after a tile's last MMA
            tc::mbar_init(&acc_empty[b], 1);  // epilogue finished reading the buffer
        }
        tc::mbar_init(mma_done, 1);
        tc::mbar_init(fix_bar, 1);
        *fix_issued = 0;
        *abort_flag = 0;
        *last_flag = 0;
        *issued = 0;
        *sfr_issued = 0;
        tc::fence_mbar_init();
        tc::tma_prefetch_desc(&tmap_w);
        if (!AQ) tc::tma_prefetch_desc(&tmap_x);
        tc::tma_prefetch_desc(&tmap_sf);
        if (A4) tc::tma_prefetch_desc(&tmap_sfb);
        if (p.tma_out) tc::tma_prefetch_desc(&tmap_out);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, L::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Raw scale tiles of 4-k-tile unit g into raw slot rs: the weight rows' [128 x 16 B] and, for
    // W4A4, the tokens' [BN x 16 B] (the caller has armed sfr_full[rs] for SFR_BYTES).
    auto load_raw_scales = [&](int g, int rs) {
        int kts, ns, mts;
        sched.fill_at(4 * g, p.m_tiles, kts, ns, mts);
        tc::tma_load_2d(smem + L::SFR_OFF + rs * L::SFR_BYTES, &tmap_sf, &sfr_full[rs], 4 * kts, ns);
        if constexpr (A4)
            tc::tma_load_2d(smem + L::SFR_OFF + rs * L::SFR_BYTES + L::SFR_B_OFF, &tmap_sfb, &sfr_full[rs], 4 * kts,
                            mts * BN);
    };

    // Unit scale (2^0) for the activation operand: 0x7F in every byte of the B-scale columns.
    if (!A4 && warp >= EPI_WARP0) {
        const uint32_t base = tmem + L::T_SFB + ((32u * (warp & 3)) << 16);
        tc::tmem_st4(base, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
        tc::tmem_st4(base + 4, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
        tc::tmem_st_wait();
    }
    // Early weights: when the kernel before this one in the stream is known to leave the weights
    // alone (the library's own activation quant, which itself waited for everything before it),
    // the first ring fill's weights and the first SFR scale tiles are requested now, while that
    // kernel still runs; the fill's activation half follows after the wait below.  One fill, not
    // the whole ring: every SM's early loads land on HBM just as the quant kernel reads its rows,
    // and a ring's worth from 150 SMs (10-20 MB) slows that kernel, which this one then waits for
    // (decode step of 8 linears on GB300: 204.4 us with every fill early, 201.6 with one, 204.5
    // with none).
    int pre = 0;  // ring fills whose weights went out early (producer thread)
    if (!A4 && p.w_early && threadIdx.x == 0) {
        for (int g = 0; g < min(n_k / 4, SFR); ++g) {
            tc::mbar_arrive_expect_tx(&sfr_full[g], L::SFR_BYTES);
            load_raw_scales(g, g);
            atomicMax(sfr_issued, g + 1);
        }
        const uint64_t w_policy = tc::make_policy_evict_first();
        for (; pre < min(n_k / KPU, 1); ++pre) {
            int kt, n0;
            sched.fill_at(pre * KPU, p.m_tiles, kt, n0);
            tc::mbar_arrive_expect_tx(&full[pre], L::TX_BYTES);  // weights now, activations later
            if (p.evict_first)
                tc::tma_load_3d_hint(smem + L::W_OFF + pre * L::W_SLOT, &tmap_w, &full[pre], 0, n0, kt, w_policy);
            else
                tc::tma_load_3d(smem + L::W_OFF + pre * L::W_SLOT, &tmap_w, &full[pre], 0, n0, kt);
            *issued = pre + 1;
        }
    }
    // programmatic dependent launch: everything above overlapped the previous kernel in the
    // stream; wait for it to complete before the first global memory access, and let the next
    // kernel start its own set-up early (it waits the same way before touching memory)
    tc::grid_dependency_wait();
    tc::grid_dependents_launch();
    tc::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) trace_phase(p, 1);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const int n_units = n_k / 4;
            const uint64_t w_policy = tc::make_policy_evict_first();
            if (!p.w_early) {
                // the first SFR units' raw scale tiles (later ones come from the scale warps)
                for (int g = 0; g < min(n_units, SFR); ++g) {
                    tc::mbar_arrive_expect_tx(&sfr_full[g], L::SFR_BYTES);
                    load_raw_scales(g, g);
                    atomicMax(sfr_issued, g + 1);
                }
            }
            for (int i = 0; i < n_k && !*abort_flag; i += KPU) {
                const long long u = sched.unit_at(i / 4);
                const int t = (int)div_nonneg(u, p.U);
                const int kt = (int)(u - (long long)t * p.U) * 4 + (i & 3);  // first k-tile of the fill
                const int n0 = (t / p.m_tiles) * BM, m0 = (t % p.m_tiles) * BN;
                const int f = i / KPU, sl = f % US;
                if (f >= pre) {
                    if (wait_or_fail(&empty[sl], ((f / US) & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER, i))
                        break;
                    tc::mbar_arrive_expect_tx(&full[sl], L::TX_BYTES);
                    if (p.evict_first)
                        tc::tma_load_3d_hint(smem + L::W_OFF + sl * L::W_SLOT, &tmap_w, &full[sl], 0, n0, kt, w_policy);
                    else
                        tc::tma_load_3d(smem + L::W_OFF + sl * L::W_SLOT, &tmap_w, &full[sl], 0, n0, kt);
                }

                // prefill tilings: every activation tile is read again by the CTAs working on
                // other weight tiles, so it is kept in L2 over the streaming weights and outputs
                // (with the fused activation quant the quantizer warps write the tiles instead)
                if constexpr (AQ)
                    ;
                else if constexpr (BN >= 128)
                    tc::tma_load_3d_hint(smem + L::X_OFF + sl * L::X_SLOT, &tmap_x, &full[sl], 0, m0, kt,
                                         tc::make_policy_evict_last());
                else
                    tc::tma_load_3d(smem + L::X_OFF + sl * L::X_SLOT, &tmap_x, &full[sl], 0, m0, kt);
                *issued = f + 1;
                trace_ev(p, TR_TMA_ISSUED, i);
                trace_ev(p, TR_TMA_FILL, f);
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
        int f = 0;
        for (int seg = 0; seg < sched.S; ++seg) {
            long long u, ue;
            sched.seg_units(seg, u, ue);
            const int b = seg % ACC_BUFS;
            const uint32_t t_acc = tmem + b * BN;
            const int f_end = f + (int)(4 * (ue - u)) / KPU;
            for (bool first = true; f < f_end; ++f, first = false) {
                const int sl = f % US;
                const int sq = f % SFQ;
                if (gate && lane == 0) {  // lane 0 waits; the named barrier releases the rest
                    if (!*abort_flag && first)
                        wait_or_fail(&acc_empty[b], ((seg / ACC_BUFS) & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_GATE, seg);
                    if (!*abort_flag) wait_or_fail(&sff[sq], (f / SFQ) & 1, abort_flag, p.status, ST_TIMEOUT_GATE, f);
                    trace_ev(p, TR_GATE_SFF, f);
                    if (!*abort_flag) wait_or_fail(&full[sl], (f / US) & 1, abort_flag, p.status, ST_TIMEOUT_GATE, f);
                    trace_ev(p, TR_MMA_READY, f);
                    if (f == 0) trace_phase(p, 8);
                    if (f == n_k / KPU - 1) trace_phase(p, 9);
                }
                // the gate's abort state rides on the barrier: the MMA thread reads no memory here
                const bool aborted = tc::named_bar_or(GATE_BARRIER, 64, gate && *abort_flag);
                if (!gate && lane == 0 && !aborted) {
                    tc::tc_fence_after();
#pragma unroll
                    for (int j = 0; j < KPU; ++j) {
                        const uint32_t sfa = tmem + L::T_SFA + 4 * (sq * KPU + j);
                        const uint32_t wa = tc::smem_u32(smem + L::W_OFF + sl * L::W_SLOT + j * L::W_TILE);
                        const uint32_t xa = tc::smem_u32(smem + L::X_OFF + sl * L::X_SLOT + j * L::X_TILE);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = tc::smem_desc(wa + 32 * kk, 16, 1024, 2);
                            const uint64_t bd = tc::smem_desc(xa + 32 * kk, 16, 1024, 2);
                            const uint32_t sfb = A4 ? tmem + L::T_SFB + L::SFBW * (sq * KPU + j) : tmem + L::T_SFB;
                            tc::mma_mxf8f6f4(t_acc, ad, bd, tc::idesc_mxf8f6f4(5, A4 ? 5 : 0, BM, BN, kk, A4 ? kk : 0),
                                             sfa, sfb, (first && j == 0 && kk == 0) ? 0u : 1u);
                        }
                    }
                    tc::tc_commit(&empty[sl]);
                    if (SFQ != US) tc::tc_commit(&sfe[sq]);
                    if (f_end - f == 1) tc::tc_commit(&acc_full[b]);
                }
                __syncwarp();
            }
        }
        if (!gate && lane == 0) {
            tc::tc_commit(mma_done);  // teardown waits on it before freeing TMEM
            trace_phase(p, 10);
        }
        __syncwarp();
    } else if (warp < EPI_WARP0) {
        // ------------------------------------------------------------ scale warps (2-5)
        // Warp w owns TMEM lanes 32q..32q+31, q = w & 3 (weight rows 32q..32q+31).  For each
        // k-tile of a ring fill it writes its rows' 4-byte scale word (the 4 k-block scales of
        // that k-tile) into the 4 columns of the fill's TMEM scale slot, once the raw scale tile
        // has landed and the MMAs that last read the slot have finished; the data of the fill
        // need not have arrived, so this work stays off the path from TMA to MMA.
        const int q = warp & 3;
        const int row = 32 * q + lane;
        // Fused activation quant: thread st_t owns 4-value chunk st_t of every fill (the fill's k
        // offsets 4 st_t .. 4 st_t + 3) for each token.  It loads fill f + 2's values and rounds
        // fill f + 1's to e4m3 (the code of w4a8_act_quant) right after finishing fill f, so when
        // fill f + 1's slot frees only the stores are left; the codes go where the
        // 128-byte-swizzled TMA box would put them.
        const int st_t = threadIdx.x - SCALE_WARP0 * 32;  // 0..127
        const int aq_kb = (st_t & 31) * 4;                // byte of the k-tile row
        float *aq_s = reinterpret_cast<float *>(smem + L::AQ_OFF);
        uint2 v_next[AQ_MAX_M];
        uint32_t qc[AQ_MAX_M];
#pragma unroll
        for (int m = 0; m < AQ_MAX_M; ++m) {
            v_next[m] = make_uint2(0u, 0u);
            qc[m] = 0u;
        }
        auto load_fill = [&](int f, uint2 (&dst)[AQ_MAX_M]) {
            if (f < n_k / KPU) {
                int kt, n0;
                sched.fill_at(f * KPU, p.m_tiles, kt, n0);
#pragma unroll
                for (int m = 0; m < AQ_MAX_M; ++m)
                    if (m < p.M)
                        dst[m] = __ldg(reinterpret_cast<const uint2 *>(p.x + (size_t)m * p.K + kt * 128 + st_t * 4));
            }
        };
        if constexpr (AQ) {
            uint2 v0[AQ_MAX_M];
            load_fill(0, v0);  // in flight during the amax step
            load_fill(1, v_next);
            // every slot's activation tile starts as zeros; rows >= M are never written again
            for (int o = st_t; o < US * L::X_SLOT / 16; o += 128)
                reinterpret_cast<uint4 *>(smem + L::X_OFF)[o] = make_uint4(0u, 0u, 0u, 0u);
            aq_row_scales<8>(p.x, p.M, p.K, 128 + st_t, aq_s, reinterpret_cast<unsigned *>(aq_s + BN));
#pragma unroll
            for (int m = 0; m < AQ_MAX_M; ++m)
                if (m < p.M) qc[m] = quant4_e4m3(v0[m], aq_s[m]);
        }
        int w = 0;
        for (int i = 0; i < n_k && !w; i += KPU) {
            const int g = i >> 2, rs = g % SFR;
            if ((i & 3) == 0 &&
                (w = warp_wait(&sfr_full[rs], (g / SFR) & 1, abort_flag, p.status, ST_TIMEOUT_SCALE, g, lane)))
                break;
            const int f = i / KPU, sq = f % SFQ;
            // with one scale slot per ring slot, the slot is free when the fill's ring slot is
            if ((w = warp_wait(SFQ == US ? &empty[f % US] : &sfe[sq], ((f / SFQ) & 1) ^ 1, abort_flag, p.status,
                               ST_TIMEOUT_SCALE, f, lane)))
                break;
            tc::tc_fence_after();
            if (lane == 0 && warp == SCALE_WARP0) trace_ev(p, TR_SCALE_DATA, f);
            const uint8_t *raw = smem + L::SFR_OFF + rs * L::SFR_BYTES + row * 16;
#pragma unroll
            for (int j = 0; j < KPU; ++j) {
                const uint32_t sw = *reinterpret_cast<const uint32_t *>(raw + 4 * ((i & 3) + j));
                tc::tmem_st4(tmem + L::T_SFA + 4 * (sq * KPU + j) + ((32u * q) << 16), sw, sw, sw, sw);
            }
            if constexpr (A4) {
                // token scales: token t = lane + 32c in column c of the slot, the same in every
                // lane quarter (each warp writes its own quarter)
                const uint8_t *rawb = smem + L::SFR_OFF + rs * L::SFR_BYTES + L::SFR_B_OFF;
#pragma unroll
                for (int j = 0; j < KPU; ++j) {
                    uint32_t v[L::SFBW];
#pragma unroll
                    for (int c = 0; c < L::SFBW; ++c) {
                        const int t = lane + 32 * c;
                        v[c] = t < BN ? *reinterpret_cast<const uint32_t *>(rawb + t * 16 + 4 * ((i & 3) + j)) : 0u;
                    }
                    const uint32_t ta = tmem + L::T_SFB + L::SFBW * (sq * KPU + j) + ((32u * q) << 16);
                    tc::tmem_st4(ta, v[0], v[1], v[2], v[3]);
                    if constexpr (L::SFBW == 8) tc::tmem_st4(ta + 4, v[4], v[5], v[6], v[7]);
                }
            }
            if constexpr (AQ) {
                uint8_t *xt = smem + L::X_OFF + (f % US) * L::X_SLOT + (st_t >> 5) * L::X_TILE;  // k-tile st_t / 32
#pragma unroll
                for (int m = 0; m < AQ_MAX_M; ++m)
                    if (m < p.M)
                        *reinterpret_cast<uint32_t *>(xt + m * 128 + ((((aq_kb >> 4) ^ (m & 7)) << 4) | (aq_kb & 15))) =
                            qc[m];
                tc::fence_proxy_async_smem();  // generic writes -> visible to the tensor core
            }
            tc::tmem_st_wait();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&sff[sq]);
                if (AQ) tc::mbar_arrive(&full[f % US]);
                if (((i + KPU) & 3) == 0) tc::mbar_arrive(&sfr_empty[rs]);
                if (warp == SCALE_WARP0) trace_ev(p, TR_SCALE_DONE, f);
                if (AQ && warp == SCALE_WARP0) trace_ev(p, TR_AQ_DONE, f);
            }
            // the unit's raw tile is consumed by all four warps: one thread loads unit g + SFR's
            // tile into the same slot, so scale loads never hold up the producer's data loads
            if (((i + KPU) & 3) == 0 && warp == SCALE_WARP0 && lane == 0 && g + SFR < n_k / 4) {
                if ((w = wait_or_fail(&sfr_empty[rs], (g / SFR) & 1, abort_flag, p.status, ST_TIMEOUT_SCALE, g)) == 0) {
                    tc::mbar_arrive_expect_tx(&sfr_full[rs], L::SFR_BYTES);
                    load_raw_scales(g + SFR, rs);
                    atomicMax(sfr_issued, g + SFR + 1);
                }
            }
            w = __shfl_sync(0xffffffffu, w, 0);
            if constexpr (AQ) {  // the next fill's codes, and the values of the one after
                if (f + 1 < n_k / KPU) {
#pragma unroll
                    for (int m = 0; m < AQ_MAX_M; ++m)
                        if (m < p.M) qc[m] = quant4_e4m3(v_next[m], aq_s[m]);
                }
                load_fill(f + 2, v_next);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int first_tile = sched.t_first;
        const int row = 32 * q + lane;
        const bool issuer = (threadIdx.x == EPI_WARP0 * 32);
        int ck = 0;  // output chunks emitted (staging buffer rotation)
        if constexpr (AQ)  // the token scales, with the quantizer warps (before any tile is done)
            aq_row_scales<16>(p.x, p.M, p.K, threadIdx.x - EPI_WARP0 * 32, reinterpret_cast<float *>(smem + L::AQ_OFF),
                          reinterpret_cast<unsigned *>(smem + L::AQ_OFF) + BN);
        // Write 16 token columns (c0..c0+15 of the tile at m0, n0) of this thread's weight row.
        // With TMA stores the 128 threads stage a [16 tokens][128 rows] bf16 block in shared memory
        // and one thread stores it (out-of-range rows and tokens are clipped by the tensor map);
        // all 128 threads must call this together.
        auto emit = [&](const float (&o)[16], int c0, int m0, int n0) {
            const int n = n0 + row;
            if (p.tma_out) {
                uint16_t *stg = reinterpret_cast<uint16_t *>(smem + L::STAGE_OFF + (ck % L::NSTAGE) * L::STAGE_BYTES);
                if (ck >= L::NSTAGE) {  // the store that last used this buffer has read it
                    if (issuer) tc::bulk_wait_group_read<L::NSTAGE - 1>();
                    tc::named_bar_sync(1, 128);
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) stg[j * BM + row] = float_to_bf16_bits(o[j]);
                tc::fence_proxy_async_smem();
                tc::named_bar_sync(1, 128);
                if (issuer) {
                    if constexpr (BN >= 128)  // prefill: the output is not read again, keep L2 for operands
                        tc::tma_store_2d_hint(&tmap_out, stg, n0, m0 + c0, tc::make_policy_evict_first());
                    else
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
        for (int seg = 0; seg < sched.S; ++seg) {
            long long u, ue;
            sched.seg_units(seg, u, ue);
            const int t = (int)div_nonneg(u, p.U);
            const long long t_lo = (long long)t * p.U, t_hi = t_lo + p.U;
            const bool whole = (u == t_lo) && (ue == t_hi);
            const int b = seg % ACC_BUFS;
            const int n0 = (t / p.m_tiles) * BM, m0 = (t % p.m_tiles) * BN;
            // the tile's per-token scales, staged once in shared memory (the load overlaps the wait)
            float *xs_s = reinterpret_cast<float *>(smem + L::XS_OFF);
            const float *aq_s = reinterpret_cast<const float *>(smem + L::AQ_OFF);
            for (int i = row; i < BN; i += BM)
                xs_s[i] = (m0 + i < p.M) ? (A4 ? 1.0f : AQ ? aq_s[m0 + i] : __ldg(p.xs + m0 + i)) : 0.0f;
            int w = 0;
            if (lane == 0) w = tc::mbar_wait(&acc_full[b], (seg / ACC_BUFS) & 1, abort_flag, WAIT_BUDGET);
            w = __shfl_sync(0xffffffffu, w, 0);
            if (w && lane == 0) {
                if (w == 1) fail(p.status, ST_TIMEOUT_EPI, &acc_full[b], seg);
                *abort_flag = 1;
            }
            // all four warps leave together if any of them gave up (this also publishes xs_s)
            if (tc::named_bar_or(1, 128, w != 0)) break;
            tc::tc_fence_after();
            if (seg == 0 && threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 11);
            const bool last_seg = (seg == sched.S - 1);
            if (last_seg && threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 4);
            const uint32_t t_acc = tmem + b * BN + ((32u * q) << 16);
            float *slot = p.partials + ((size_t)cta * 2 + (t == first_tile ? 0 : 1)) * (size_t)(BM * BN);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t r[16];
                tc::tmem_ld16(t_acc + c0, r);
                tc::tmem_ld_wait();
                if (whole) {
                    if (m0 + c0 < p.M) {
                        float o[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) o[j] = __uint_as_float(r[j]) * xs_s[c0 + j];
                        emit(o, c0, m0, n0);
                    }
                } else {
                    // only the tokens that exist: the fix-up reads no column at or past M
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (m0 + c0 + j < p.M) tc::st_cg_f32(slot + (c0 + j) * BM + row, __uint_as_float(r[j]));
                }
            }
            // release the accumulator buffer to the MMA issuer
            tc::tc_fence_before();
            tc::named_bar_sync(1, 128);
            if (threadIdx.x == EPI_WARP0 * 32) tc::mbar_arrive(&acc_empty[b]);
            if (!whole) {
                // stream-K fix-up: the last contributor of tile t adds the partials in CTA order
                const int c_first = unit_owner(t_lo, p.RU, p.Gsk);
                const int c_last = unit_owner(t_hi - 1, p.RU, p.Gsk);
                if (last_seg && threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 5);
                // the CTA's partial stores happen before one thread's acq_rel arrival (release);
                // the last arrival's acquire makes every contributor's partial visible to it
                tc::named_bar_sync(1, 128);
                if (threadIdx.x == EPI_WARP0 * 32) {
                    const int old = tc::atomic_add_acq_rel_gpu(p.counters + t, 1);
                    *last_flag = (old == c_last - c_first);
                }
                tc::named_bar_sync(1, 128);
                if (last_seg && threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 6);
                if (*last_flag) {
                    const int n_contrib = c_last - c_first + 1;
                    const int m_cnt = min(BN, p.M - m0);
                    const uint32_t part_bytes = (uint32_t)m_cnt * BM * 4;  // first m_cnt columns of a slot
                    // The CTA's last tile: every ring fill has been consumed (its accumulator is
                    // complete), so the ring's shared memory is idle.  Bulk copies bring all the
                    // contributors' partials in one round trip instead of one per 16 columns.
                    // Up to 16 tokens the plain loads below take one round trip too, without the
                    // proxy fence and the bulk copy's longer latency.
                    if (last_seg && m_cnt > 16 && (size_t)n_contrib * part_bytes <= (size_t)L::SFR_OFF) {
                        if (threadIdx.x == EPI_WARP0 * 32) {
                            tc::fence_proxy_async_global();  // partials were written by generic stores
                            tc::mbar_arrive_expect_tx(fix_bar, (uint32_t)n_contrib * part_bytes);
                            *fix_issued = 1;
                            for (int c = c_first; c <= c_last; ++c) {
                                const int sl = (t == (int)(unit_start(c, p.RU, p.Gsk) / p.U)) ? 0 : 1;
                                tc::bulk_load(smem + (size_t)(c - c_first) * part_bytes,
                                              p.partials + ((size_t)c * 2 + sl) * (size_t)(BM * BN), part_bytes, fix_bar);
                            }
                        }
                        int w = 0;
                        if (lane == 0) w = tc::mbar_wait(fix_bar, 0, abort_flag, WAIT_BUDGET);
                        w = __shfl_sync(0xffffffffu, w, 0);
                        if (threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 12);
                        if (w) {
                            if (lane == 0) {
                                if (w == 1) fail(p.status, ST_TIMEOUT_EPI, fix_bar, seg);
                                *abort_flag = 1;
                            }
                        } else {
                            // same order of additions as below: zero, then the contributors in CTA
                            // order; 16 independent columns per step keep the loads pipelined
                            const float *st = reinterpret_cast<const float *>(smem) + row;
                            const int stride = m_cnt * BM;
                            for (int c0 = 0; c0 < m_cnt; c0 += 16) {
                                float a[16];
#pragma unroll
                                for (int j = 0; j < 16; ++j) a[j] = 0.0f;
                                for (int c = 0; c < n_contrib; ++c) {
                                    const float *sc = st + c * stride + c0 * BM;
#pragma unroll
                                    for (int j = 0; j < 16; ++j)
                                        if (c0 + j < m_cnt) a[j] += sc[j * BM];
                                }
#pragma unroll
                                for (int j = 0; j < 16; ++j) a[j] *= xs_s[c0 + j];
                                if (c0 == 0 && threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 14);
                                emit(a, c0, m0, n0);
                                if (c0 == 0 && threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 15);
                            }
                        }
                        if (threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 13);
                    } else if (narrow_fixup<BN>(n_contrib)) {
                        // decode tiles: a group of contributors' whole partials per round trip (one
                        // 64-column partial, three of 32 columns, six of 16) instead of one round
                        // trip per 16-column chunk; the additions run in CTA order as below
                        constexpr int NT = BN <= 64 ? BN : 16;                     // columns held
                        constexpr int GC = BN >= 64 ? 1 : (BN <= 64 ? 96 / NT : 1);  // contributors per trip
                        float acc[NT];
#pragma unroll
                        for (int j = 0; j < NT; ++j) acc[j] = 0.0f;
                        for (int cb = c_first; cb <= c_last; cb += GC) {
                            float v[GC][NT];
#pragma unroll
                            for (int cc = 0; cc < GC; ++cc) {
                                const int c = min(cb + cc, c_last);  // past the end: reload the last, unused
                                const int sl = (t == (int)(unit_start(c, p.RU, p.Gsk) / p.U)) ? 0 : 1;
                                const float *src = p.partials + ((size_t)c * 2 + sl) * (size_t)(BM * BN) + row;
#pragma unroll
                                for (int j = 0; j < NT; ++j) v[cc][j] = j < m_cnt ? __ldcg(src + j * BM) : 0.0f;
                            }
#pragma unroll
                            for (int cc = 0; cc < GC; ++cc)
                                if (cb + cc <= c_last) {
#pragma unroll
                                    for (int j = 0; j < NT; ++j) acc[j] += v[cc][j];
                                }
                        }
#pragma unroll
                        for (int c0 = 0; c0 < NT; c0 += 16) {
                            if (c0 < m_cnt) {
                                float o[16];
#pragma unroll
                                for (int j = 0; j < 16; ++j) o[j] = acc[c0 + j] * xs_s[c0 + j];
                                emit(o, c0, m0, n0);
                            }
                        }
                    } else {
                        // 16 columns at a time, up to 6 contributors' loads in flight together; the
                        // additions still run in CTA order, so the result does not depend on timing
                        for (int c0 = 0; c0 < m_cnt; c0 += 16) {
                            float acc[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
                            for (int cb = c_first; cb <= c_last; cb += 6) {
                                float v[6][16];
#pragma unroll
                                for (int cc = 0; cc < 6; ++cc) {
                                    const int c = min(cb + cc, c_last);  // past the end: reload the last, unused
                                    const int sl = (t == (int)(unit_start(c, p.RU, p.Gsk) / p.U)) ? 0 : 1;
                                    const float *src = p.partials + ((size_t)c * 2 + sl) * (size_t)(BM * BN) + c0 * BM + row;
#pragma unroll
                                    for (int j = 0; j < 16; ++j) v[cc][j] = c0 + j < m_cnt ? __ldcg(src + j * BM) : 0.0f;
                                }
#pragma unroll
                                for (int cc = 0; cc < 6; ++cc)
                                    if (cb + cc <= c_last) {
#pragma unroll
                                        for (int j = 0; j < 16; ++j) acc[j] += v[cc][j];
                                    }
                            }
#pragma unroll
                            for (int j = 0; j < 16; ++j) acc[j] *= xs_s[c0 + j];
                            emit(acc, c0, m0, n0);
                        }
                    }
                    if (threadIdx.x == EPI_WARP0 * 32) p.counters[t] = 0;
                }
                tc::named_bar_sync(1, 128);  // last_flag is reused by the next tile
                if (last_seg && threadIdx.x == EPI_WARP0 * 32) trace_phase(p, 7);
            }
        }
        if (issuer) {
            tc::bulk_wait_group_all();  // output stores done before the CTA's shared memory goes away
            trace_phase(p, 2);
        }
    }


    tc::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        int zero = 0;
        if (*abort_flag) {
            // drain: TMA copies issued but not waited for
            for (int f = max(0, *issued - US); f < *issued; ++f)
                if (tc::mbar_wait(&full[f % US], (f / US) & 1, &zero, DRAIN_BUDGET)) break;
            for (int g = max(0, *sfr_issued - SFR); g < *sfr_issued; ++g)
                tc::mbar_wait(&sfr_full[g % SFR], (g / SFR) & 1, &zero, DRAIN_BUDGET);
            if (*fix_issued) tc::mbar_wait(fix_bar, 0, &zero, DRAIN_BUDGET);
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
    long long TU, RU;
    int R, D, Gsk;
};

// Token-tile width for M > 128, from measurements on GB300 (gate_up, down and qkv at M = 512 to
// 4096).  A 256-token tile has one accumulator (two do not fit in tensor memory beside the scale
// slots), so its epilogue does not overlap the next tile's MMAs; that pays off only over a long K.
// 224-token tiles keep two accumulators (448 columns) with almost the same reuse of each weight
// tile, and win for large M at shorter K (gate_up / qkv at M = 4096: +13% / +24% over 256).
// Below that, 192-token tiles (two accumulators) are fastest when there are at least five per
// CTA, and 128-token tiles, which spread better over the SMs, below that.
static int prefill_bn(int64_t M, int64_t N, int64_t K)
{
    if (K >= 16384) return M > 1024 ? 256 : 128;
    if (M >= 3072) return 224;
    const long long n_tiles = (N + BM - 1) / BM;
    return n_tiles * ((M + 191) / 192) >= 5ll * tch::num_sms() ? 192 : 128;
}

Cfg choose(int64_t M, int64_t N, int64_t K)
{
    Cfg c;
    c.BN = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : prefill_bn(M, N, K);
    c.n_tiles = (int)((N + BM - 1) / BM);
    c.m_tiles = (int)((M + c.BN - 1) / c.BN);
    c.U = (int)(K / 512);
    c.TU = (long long)c.n_tiles * c.m_tiles * c.U;
    c.G = (int)std::min<long long>(tch::num_sms(), c.TU);
    const int T = c.n_tiles * c.m_tiles;
    c.D = T / c.G;        // whole tiles per CTA
    c.R = T - c.D * c.G;  // tiles split stream-K over all CTAs
    c.RU = (long long)c.R * c.U;
    c.Gsk = (int)std::max<long long>(1, std::min<long long>(c.G, c.RU));
    return c;
}

size_t partial_bytes(const Cfg &c)
{
    size_t b = (size_t)c.G * 2 * BM * c.BN * 4;
    return (b + 255) / 256 * 256;
}

size_t workspace_for(const Cfg &c)
{
    return W4A8_COUNTER_BYTES + partial_bytes(c);
}

template <int BN, int KPU, int US, int ACC_BUFS, int SFQ, int SFR, bool A4 = false, bool AQ = false>
w4a8_status launch(const uint8_t *wp, const uint8_t *xq, Params prm, cudaStream_t stream,
                   const uint8_t *xe = nullptr)
{
    using L = Layout<BN, KPU, US, ACC_BUFS, SFQ, SFR, A4, AQ>;
    CUtensorMap tw, tx, tsf, tout, tsfb;
    memset(&tsfb, 0, sizeof(tsfb));
    memset(&tx, 0, sizeof(tx));
    // W4A4: activations are 4-bit codes [M, K/2] read like the weights, their e8m0 [M, K/32] as
    // [BN tokens x 16 bytes] tiles
    if (A4 && (!tch::tmap_3d_ktiles(&tx, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, xq, prm.M, prm.K / 2, 64,
                                    prm.K / 128, BN, KPU) ||
               !tch::tmap_2d(&tsfb, CU_TENSOR_MAP_DATA_TYPE_UINT8, xe, prm.M, prm.K / 32, prm.K / 32, BN, 16,
                             CU_TENSOR_MAP_SWIZZLE_NONE)))
        return W4A8_ERR_CUDA;
    // output through TMA when its rows are 16-byte strided and the base 16-byte aligned
    memset(&tout, 0, sizeof(tout));
    prm.tma_out = (prm.N % 8 == 0) && w4a8_aligned(prm.out, 16) &&
                  tch::tmap_2d(&tout, CU_TENSOR_MAP_DATA_TYPE_UINT16, prm.out, prm.M, prm.N, (uint64_t)prm.N * 2, 16,
                               BM, CU_TENSOR_MAP_SWIZZLE_NONE);
    // 3-D views [k-tile][row][128 K]: weights (4-bit codes; a row is K/2 bytes, a k-tile 64) and
    // activations (bytes; a row is K bytes, a k-tile 128)
    if (!tch::tmap_3d_ktiles(&tw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, wp, prm.N, prm.K / 2, 64, prm.K / 128, BM,
                             KPU) ||
        (!A4 && !AQ && !tch::tmap_3d_ktiles(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, prm.M, prm.K, 128, prm.K / 128, BN, KPU)) ||
        !tch::tmap_2d(&tsf, CU_TENSOR_MAP_DATA_TYPE_UINT8, prm.we, prm.N, prm.K / 32, prm.K / 32, BM, 16,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
        return W4A8_ERR_CUDA;
    auto kern = mxfp4_tc_kernel<BN, KPU, US, ACC_BUFS, SFQ, SFR, A4, AQ>;
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
    if (cudaLaunchKernelEx(&cfg, kern, tw, tx, tsf, tout, tsfb, prm) != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
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

size_t w4a8_tc_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (K % 512 != 0 || K <= 0 || M <= 0 || N <= 0) return 0;
    return workspace_for(choose(M, N, K));
}

static bool make_params(Params &prm, const Cfg &c, const float *x_scale, const uint8_t *wp, const uint8_t *we,
                        uint16_t *out, int64_t M, int64_t N, int64_t K, void *workspace, bool w_early)
{
    prm.wp = wp;
    prm.we = we;
    prm.xs = x_scale;
    prm.x = nullptr;
    prm.out = out;
    if (c.G > W4A8_MAX_COUNTERS) return false;  // split tiles are indexed below the grid size
    prm.counters = static_cast<int *>(workspace);
    prm.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + W4A8_COUNTER_BYTES);
    prm.status = w4a8_device_status_ptr();
    prm.M = (int)M;
    prm.N = (int)N;
    prm.K = (int)K;
    prm.m_tiles = c.m_tiles;
    prm.n_tiles = c.n_tiles;
    prm.U = c.U;
    prm.RU = c.RU;
    prm.R = c.R;
    prm.D = c.D;
    prm.Gsk = c.Gsk;
    prm.G = c.G;
    prm.trace = static_cast<unsigned long long *>(w4a8_debug_trace_ptr());
    // a single token tile reads every weight once: keep it from displacing other lines in L2
    prm.evict_first = c.m_tiles == 1;
    prm.w_early = w_early ? 1 : 0;
    return prm.status != nullptr;
}

w4a8_status w4a8_launch_mxfp4_tc(const uint8_t *xq, const float *x_scale, const uint8_t *wp, const uint8_t *we,
                                 uint16_t *out, int64_t M, int64_t N, int64_t K, void *workspace, int,
                                 bool w_early, cudaStream_t stream)
{
    const Cfg c = choose(M, N, K);
    Params prm;
    if (!make_params(prm, c, x_scale, wp, we, out, M, N, K, workspace, w_early)) return W4A8_ERR_CUDA;
    switch (c.BN) {
    case 16: return launch<16, 4, 3, 2, 3, 2>(wp, xq, prm, stream);
    case 32: return launch<32, 4, 2, 2, 2, 4>(wp, xq, prm, stream);
    case 64: return launch<64, 4, 2, 2, 2, 4>(wp, xq, prm, stream);
    case 128: return launch<128, 2, 3, 2, 6, 4>(wp, xq, prm, stream);
    case 192: return launch<192, 2, 2, 2, 2, 4>(wp, xq, prm, stream);
    case 224: return launch<224, 2, 2, 2, 2, 4>(wp, xq, prm, stream);
    default: return launch<256, 2, 2, 1, 4, 4>(wp, xq, prm, stream);
    }
}

bool w4a8_tc_mxfp4_aq_takes(int64_t M, int64_t K)
{
    return M >= 1 && M <= AQ_MAX_M && (size_t)M * (size_t)K * 2 <= W4A8_FUSED_AQ_MAX_X_BYTES;
}

w4a8_status w4a8_launch_mxfp4_tc_aq(const uint16_t *x_bf16, const uint8_t *wp, const uint8_t *we, uint16_t *out,
                                    int64_t M, int64_t N, int64_t K, void *workspace, cudaStream_t stream)
{
    const Cfg c = choose(M, N, K);  // M <= AQ_MAX_M: the 16-token tiling
    Params prm;
    if (!make_params(prm, c, nullptr, wp, we, out, M, N, K, workspace, false)) return W4A8_ERR_CUDA;
    prm.x = x_bf16;
    return launch<16, 4, 3, 2, 3, 2, false, true>(wp, nullptr, prm, stream);
}

bool w4a8_tc_mxfp4_a4_supported(const void *xa, const void *xe, const void *wp, const void *we, const void *out,
                                int64_t M, int64_t N, int64_t K)
{
    // the activation codes are read like the weights (32-byte aligned), their scales like the weights'
    return w4a8_tc_mxfp4_supported(xa, wp, we, out, M, N, K) && w4a8_aligned(xa, 32) && w4a8_aligned(xe, 16);
}

w4a8_status w4a8_launch_mxfp4_a4_tc(const uint8_t *xa, const uint8_t *xe, const uint8_t *wp, const uint8_t *we,
                                    uint16_t *out, int64_t M, int64_t N, int64_t K, void *workspace, int,
                                    cudaStream_t stream)
{
    const Cfg c = choose(M, N, K);
    Params prm;
    if (!make_params(prm, c, nullptr, wp, we, out, M, N, K, workspace, false)) return W4A8_ERR_CUDA;
    switch (c.BN) {
    case 16: return launch<16, 4, 3, 2, 3, 2, true>(wp, xa, prm, stream, xe);
    case 32: return launch<32, 4, 2, 2, 2, 4, true>(wp, xa, prm, stream, xe);
    case 64: return launch<64, 4, 2, 2, 2, 4, true>(wp, xa, prm, stream, xe);
    case 128: return launch<128, 2, 3, 2, 6, 4, true>(wp, xa, prm, stream, xe);
    case 192: return launch<192, 2, 2, 2, 2, 4, true>(wp, xa, prm, stream, xe);
    case 224: return launch<224, 2, 2, 2, 2, 4, true>(wp, xa, prm, stream, xe);
    default: return launch<256, 2, 2, 1, 4, 3, true>(wp, xa, prm, stream, xe);
    }
}
