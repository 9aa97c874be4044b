// gemm_tc.cu -- tensor-core (tcgen05, sm_103a) MXFP4 W4A8 GEMM.
//
// "vllm-radiance (MXFP4)", "The W4A8 fp8-WMMA kernel": fp8 (e4m3) activations times e2m1
// weights with the e8m0 block scale folded into the matrix instruction, a prefill tiling and
// a decode tiling whose split-K partials are reduced by the last CTA to arrive (no second
// launch).  The pages' kernel is an RDNA4 WMMA design; this one is built for Blackwell:
//
//   * swap-AB: the weights are the MMA "M" operand (128 weight rows per tile) and the tokens
//     the "N" operand (16..256), so a decode batch of 1-64 tokens still fills the instruction;
//   * tcgen05.mma kind::mxf8f6f4 with block_scale.scale_vec::1X: A = e2m1 weights with their
//     ue8m0 scale per 32 along K, B = e4m3 activations with a unit scale (0x7F), fp32
//     accumulator in tensor memory; the per-token scale is applied in the epilogue;
//   * weights reach shared memory through TMA in the 16U4_ALIGN16B form (each 16 packed e2m1
//     codes land in a 16-byte slot, the layout the f8f6f4 instruction reads for 4-bit
//     operands), activations through TMA as bytes, both with the 128-byte swizzle;
//   * the weight scales of each stage are staged by a helper warp into a 128 x 16-byte block
//     (row r holds its 4-byte scale word four times) and copied to tensor memory with
//     tcgen05.cp, so lane r of every scale column holds row r's word;
//   * warp roles: warp 0 TMA producer, warp 1 TMEM allocator + MMA issuer, warp 2 scale
//     staging, warps 3-6 epilogue (each reads the TMEM lane quarter its warp index selects).
//
// Every mbarrier wait is bounded; a wait that gives up sets a bit in the library's device
// status word, the CTA drains what it started and returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "dispatch.h"
#include "tc_ptx.cuh"

namespace w4a8 {
namespace tcg {

constexpr int BM = 128;            // weight rows per tile (MMA M)
constexpr int BK = 128;            // K elements per pipeline stage
constexpr int NUM_THREADS = 224;   // 7 warps
constexpr int EPI_WARP0 = 3;
constexpr long long WAIT_BUDGET = 1ll << 29;  // clock cycles (a quarter second or so)
constexpr long long DRAIN_BUDGET = 1ll << 24;
constexpr int SF_PREFETCH = 8;     // k-tiles of scale words kept in flight by the staging warp

enum : unsigned { ST_TIMEOUT_PRODUCER = 1, ST_TIMEOUT_MMA = 2, ST_TIMEOUT_SF = 4, ST_TIMEOUT_EPI = 8 };

struct Params {
    const uint8_t *we;     // [N, K/32] e8m0
    const float *xs;       // [M] per-token scale
    uint16_t *out;         // [M, N] bf16
    float *partials;       // [KS, M, N] fp32 split-K partials (KS > 1)
    int *counters;         // [m_tiles * n_tiles] arrival counters (KS > 1)
    unsigned int *status;  // device status word
    int M, N, K, KS, KT;
};

template <int BN, int STAGES>
struct Layout {
    static constexpr int W_BYTES = BM * 128;   // 128 rows x 128 K, 4-bit codes in 16-byte slots
    // The transaction count of a 16U4_ALIGN16B tile is the packed bytes read from global memory
    // (64 per row), not its padded shared-memory footprint.
    static constexpr int W_TX_BYTES = BM * 64;
    static constexpr int X_BYTES = BN * 128;   // BN tokens x 128 K bytes
    static constexpr int SF_BYTES = BM * 16;   // 128 rows x (scale word x 4)
    static constexpr int W_OFF = 0;
    static constexpr int X_OFF = W_OFF + STAGES * W_BYTES;
    static constexpr int SF_OFF = X_OFF + STAGES * X_BYTES;
    static constexpr int SFR_SLOTS = 2;        // raw scale tiles (128 rows x 16 bytes = 4 k-tiles)
    static constexpr int SFR_BYTES = BM * 16;
    static constexpr int SFR_OFF = SF_OFF + STAGES * SF_BYTES;
    static constexpr int BAR_OFF = SFR_OFF + SFR_SLOTS * SFR_BYTES;
    static constexpr int TOTAL = BAR_OFF + 256 + 1024;  // barriers, flags, alignment slack
    static constexpr int TMEM_NEED = BN + 8 + 4 * STAGES;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64
                                     : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
    static_assert(TMEM_NEED <= 512, "tensor memory");
    static_assert(TOTAL <= 232448, "shared memory");
};

// Record a bounded wait that ran out: the role's bit in word 0 of the status block; the first
// such event also leaves the barrier's raw state (words 2-3) and the loop index (word 1).
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

// SF_TMA: the weight scales of 4 consecutive k-tiles arrive as one [128 rows x 16 bytes] TMA
// tile (needs K a multiple of 512 so the scale rows are 16-byte strided, and split boundaries
// on multiples of 4 k-tiles); otherwise the staging warp reads them with plain loads.
template <int BN, int STAGES, bool SF_TMA>
__global__ void __launch_bounds__(NUM_THREADS, 1)
mxfp4_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_sf, const Params p)
{
    using L = Layout<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *empty = full + STAGES;
    uint64_t *accf = empty + STAGES;
    uint64_t *sfr_full = accf + 1;
    uint64_t *sfr_empty = sfr_full + L::SFR_SLOTS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sfr_empty + L::SFR_SLOTS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *last_flag = reinterpret_cast<int *>(tmem_slot + 2);
    int *consumed = reinterpret_cast<int *>(tmem_slot + 3);
    int *issued = reinterpret_cast<int *>(tmem_slot + 4);
    int *sfr_issued = reinterpret_cast<int *>(tmem_slot + 5);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BM, m0 = blockIdx.y * BN, split = blockIdx.z;
    // split boundaries: whole groups of 4 k-tiles when the scales come by TMA
    const int unit = SF_TMA ? 4 : 1;
    const int n_units = p.KT / unit;
    const int kt_begin = unit * (int)((long long)split * n_units / p.KS);
    const int kt_end = unit * (int)((long long)(split + 1) * n_units / p.KS);
    const int nkt = kt_end - kt_begin;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(&full[s], 2);   // producer expect_tx + scale-staging warp
            tc::mbar_init(&empty[s], 1);  // tcgen05.commit of the stage's MMAs
        }
        tc::mbar_init(accf, 1);
        for (int r = 0; r < L::SFR_SLOTS; ++r) {
            tc::mbar_init(&sfr_full[r], 1);
            tc::mbar_init(&sfr_empty[r], 1);
        }
        *abort_flag = 0;
        *last_flag = 0;
        *consumed = 0;
        *issued = 0;
        *sfr_issued = 0;
        tc::fence_mbar_init();
        tc::tma_prefetch_desc(&tmap_w);
        tc::tma_prefetch_desc(&tmap_x);
        if (SF_TMA) tc::tma_prefetch_desc(&tmap_sf);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, L::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_acc = tmem;
    const uint32_t t_sfb = tmem + BN;
    const uint32_t t_sfa = tmem + BN + 8;

    // Unit scale (2^0) for the activation operand: 0x7F in every byte of the B-scale columns.
    if (warp >= EPI_WARP0) {
        const uint32_t q = warp & 3;
        const uint32_t base = t_sfb + ((32u * q) << 16);
        tc::tmem_st4(base, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
        tc::tmem_st4(base + 4, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
        tc::tmem_st_wait();
    }
    tc::tc_fence_before();
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int i = 0; i < nkt; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (i / STAGES) & 1;
                if (SF_TMA && (i & 3) == 0) {
                    const int g = i >> 2, rs = g % L::SFR_SLOTS;
                    const int w = tc::mbar_wait(&sfr_empty[rs], ((g / L::SFR_SLOTS) & 1) ^ 1, abort_flag, WAIT_BUDGET);
                    if (w) {
                        if (w == 1) fail(p.status, ST_TIMEOUT_PRODUCER, &sfr_empty[rs], i);
                        *abort_flag = 1;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(&sfr_full[rs], L::SFR_BYTES);
                    tc::tma_load_2d(smem + L::SFR_OFF + rs * L::SFR_BYTES, &tmap_sf, &sfr_full[rs],
                                    4 * (kt_begin + i), n0);
                    *sfr_issued = g + 1;
                }
                const int w = tc::mbar_wait(&empty[s], ph ^ 1, abort_flag, WAIT_BUDGET);
                if (w) {
                    if (w == 1) fail(p.status, ST_TIMEOUT_PRODUCER, &empty[s], i);
                    *abort_flag = 1;
                    break;
                }
                tc::mbar_arrive_expect_tx(&full[s], L::W_TX_BYTES + L::X_BYTES);
                const int k = (kt_begin + i) * BK;
                tc::tma_load_2d(smem + L::W_OFF + s * L::W_BYTES, &tmap_w, &full[s], k, n0);
                tc::tma_load_2d(smem + L::X_OFF + s * L::X_BYTES, &tmap_x, &full[s], k, m0);
                *issued = i + 1;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            tc::tc_fence_after();
            for (int i = 0; i < nkt; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (i / STAGES) & 1;
                const int w = tc::mbar_wait(&full[s], ph, abort_flag, WAIT_BUDGET);
                if (w) {
                    if (w == 1) fail(p.status, ST_TIMEOUT_MMA, &full[s], i);
                    *abort_flag = 1;
                    break;
                }
                *consumed = i + 1;
                tc::tc_fence_after();
                const uint32_t sfa = t_sfa + 4 * s;
                tc::tc_cp_128x128b(sfa, tc::smem_desc(tc::smem_u32(smem + L::SF_OFF + s * L::SF_BYTES), 128, 128, 0));
                const uint32_t wa = tc::smem_u32(smem + L::W_OFF + s * L::W_BYTES);
                const uint32_t xa = tc::smem_u32(smem + L::X_OFF + s * L::X_BYTES);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = tc::smem_desc(wa + 32 * kk, 16, 1024, 2);
                    const uint64_t bd = tc::smem_desc(xa + 32 * kk, 16, 1024, 2);
                    tc::mma_mxf8f6f4(t_acc, ad, bd, tc::idesc_mxf8f6f4(5, 0, BM, BN, kk, 0), sfa, t_sfb,
                                     (i | kk) != 0);
                }
                tc::tc_commit(&empty[s]);
            }
            tc::tc_commit(accf);  // always: the epilogue / teardown wait on it
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ scale staging
        if constexpr (SF_TMA) {
            bool ok = true;
            for (int g = 0; 4 * g < nkt && ok; ++g) {
                const int rs = g % L::SFR_SLOTS;
                int w = 0;
                if (lane == 0) w = tc::mbar_wait(&sfr_full[rs], (g / L::SFR_SLOTS) & 1, abort_flag, WAIT_BUDGET);
                w = __shfl_sync(0xffffffffu, w, 0);
                if (w) {
                    if (lane == 0) {
                        if (w == 1) fail(p.status, ST_TIMEOUT_SF, &sfr_full[rs], g);
                        *abort_flag = 1;
                    }
                    break;
                }
                const uint8_t *raw = smem + L::SFR_OFF + rs * L::SFR_BYTES;
                for (int t = 0; t < 4; ++t) {
                    const int i = 4 * g + t;
                    if (i >= nkt) break;
                    const int s = i % STAGES;
                    w = 0;
                    if (lane == 0) w = tc::mbar_wait(&empty[s], ((i / STAGES) & 1) ^ 1, abort_flag, WAIT_BUDGET);
                    w = __shfl_sync(0xffffffffu, w, 0);
                    if (w) {
                        if (lane == 0) {
                            if (w == 1) fail(p.status, ST_TIMEOUT_SF, &empty[s], i);
                            *abort_flag = 1;
                        }
                        ok = false;
                        break;
                    }
                    uint8_t *dst = smem + L::SF_OFF + s * L::SF_BYTES;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int row = lane + 32 * r;
                        const uint32_t v = *reinterpret_cast<const uint32_t *>(raw + row * 16 + 4 * t);
                        *reinterpret_cast<uint4 *>(dst + row * 16) = make_uint4(v, v, v, v);
                    }
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&full[s]);
                }
                __syncwarp();
                if (lane == 0 && ok) tc::mbar_arrive(&sfr_empty[rs]);
            }
        } else {
            const int kb_row = p.K / 32;
            uint32_t ring[SF_PREFETCH][4];
            auto load = [&](int kt, uint32_t(&w)[4]) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int n = n0 + lane + 32 * r;
                    w[r] = n < p.N ? __ldg(reinterpret_cast<const uint32_t *>(p.we + (size_t)n * kb_row + 4 * kt))
                                   : 0x7f7f7f7fu;
                }
            };
#pragma unroll
            for (int j = 0; j < SF_PREFETCH; ++j)
                if (j < nkt) load(kt_begin + j, ring[j]);
            bool ok = true;
            for (int base = 0; base < nkt && ok; base += SF_PREFETCH) {
#pragma unroll
                for (int j = 0; j < SF_PREFETCH; ++j) {
                    const int i = base + j;
                    if (i >= nkt) break;
                    const int s = i % STAGES;
                    const uint32_t ph = (i / STAGES) & 1;
                    int w = 0;
                    if (lane == 0) w = tc::mbar_wait(&empty[s], ph ^ 1, abort_flag, WAIT_BUDGET);
                    w = __shfl_sync(0xffffffffu, w, 0);
                    if (w) {
                        if (lane == 0) {
                            if (w == 1) fail(p.status, ST_TIMEOUT_SF, &empty[s], i);
                            *abort_flag = 1;
                        }
                        ok = false;
                        break;
                    }
                    uint8_t *dst = smem + L::SF_OFF + s * L::SF_BYTES;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const uint32_t w = ring[j][r];
                        *reinterpret_cast<uint4 *>(dst + (lane + 32 * r) * 16) = make_uint4(w, w, w, w);
                    }
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&full[s]);
                    if (i + SF_PREFETCH < nkt) load(kt_begin + i + SF_PREFETCH, ring[j]);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int n = n0 + 32 * q + lane;
        int w = 0;
        if (lane == 0) w = tc::mbar_wait(accf, 0, abort_flag, WAIT_BUDGET);
        w = __shfl_sync(0xffffffffu, w, 0);
        if (w == 0 && !*abort_flag) {
            tc::tc_fence_after();
            const uint32_t row_addr = t_acc + ((32u * q) << 16);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t r[16];
                tc::tmem_ld16(row_addr + c0, r);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int m = m0 + c0 + j;
                    if (m < p.M && n < p.N) {
                        const float v = __uint_as_float(r[j]);
                        if (p.KS == 1)
                            p.out[(size_t)m * p.N + n] = float_to_bf16_bits(v * __ldg(p.xs + m));
                        else
                            p.partials[((size_t)split * p.M + m) * p.N + n] = v;
                    }
                }
            }
            if (p.KS > 1) {
                __threadfence();
                tc::named_bar_sync(1, 128);
                const int tile = blockIdx.y * gridDim.x + blockIdx.x;
                if (threadIdx.x == EPI_WARP0 * 32) {
                    const int old = atomicAdd(p.counters + tile, 1);
                    *last_flag = (old == p.KS - 1);
                }
                tc::named_bar_sync(1, 128);
                if (*last_flag) {
                    __threadfence();
                    if (n < p.N) {
                        const int m_end = min(m0 + BN, p.M);
                        for (int m = m0; m < m_end; ++m) {
                            float acc = 0.0f;
                            for (int z = 0; z < p.KS; ++z)
                                acc += __ldcg(p.partials + ((size_t)z * p.M + m) * p.N + n);
                            p.out[(size_t)m * p.N + n] = float_to_bf16_bits(acc * __ldg(p.xs + m));
                        }
                    }
                    if (threadIdx.x == EPI_WARP0 * 32) p.counters[tile] = 0;
                }
            }
        } else if (lane == 0 && w) {
            if (w == 1) fail(p.status, ST_TIMEOUT_EPI, accf, 0);
            *abort_flag = 1;
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        // drain: TMA copies issued but not consumed, and the MMAs behind the final commit
        int zero = 0;
        for (int i = *consumed; i < *issued; ++i)
            if (tc::mbar_wait(&full[i % STAGES], (i / STAGES) & 1, &zero, DRAIN_BUDGET)) break;
        for (int g = max(0, *sfr_issued - L::SFR_SLOTS); g < *sfr_issued; ++g)
            tc::mbar_wait(&sfr_full[g % L::SFR_SLOTS], (g / L::SFR_SLOTS) & 1, &zero, DRAIN_BUDGET);
        tc::mbar_wait(accf, 0, &zero, WAIT_BUDGET);
    }
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// ------------------------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

bool tmap_w_fp4(CUtensorMap *m, const void *w, int64_t N, int64_t K)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {128, (cuuint32_t)BM};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void *>(w), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tmap_bytes(CUtensorMap *m, const void *x, int64_t rows, int64_t cols, int box_rows, int box_cols,
                CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(x), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms()
{
    static int cache[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!cache[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = v > 0 ? v : 148;
    }
    return cache[dev];
}

struct Cfg {
    int BN, KS, m_tiles, n_tiles;
    bool sf_tma;
};

Cfg choose(int64_t M, int64_t N, int64_t K)
{
    Cfg c;
    c.BN = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
    c.n_tiles = (int)((N + BM - 1) / BM);
    c.m_tiles = (int)((M + c.BN - 1) / c.BN);
    const int KT = (int)(K / BK);
    c.sf_tma = (K % 512) == 0;
    const int units = c.sf_tma ? KT / 4 : KT;  // split granularity
    const long long tiles = (long long)c.n_tiles * c.m_tiles;
    const int sms = num_sms();
    c.KS = 1;
    if (tiles < 2LL * sms) {
        // split K so the grid fills the SMs evenly; fp32 partials cost traffic, so weigh
        // their bytes (written and read back, mostly in L2) against the weight bytes
        double best = -1e30;
        const double wbytes = (double)N * K * 17.0 / 32.0;
        for (int ks = 1; ks <= units && ks <= 32; ++ks) {
            const long long ctas = tiles * ks;
            const long long waves = (ctas + sms - 1) / sms;
            const double eff = (double)ctas / (double)(waves * sms);
            const double part = ks > 1 ? 8.0 * ks * (double)M * N / wbytes : 0.0;
            const double score = eff - 0.25 * part - 0.002 * ks;
            if (score > best) {
                best = score;
                c.KS = ks;
            }
        }
    }
    return c;
}

size_t workspace_for(const Cfg &c, int64_t M, int64_t N)
{
    if (c.KS <= 1) return 0;
    size_t part = (size_t)c.KS * (size_t)M * (size_t)N * 4;
    part = (part + 255) / 256 * 256;
    return part + (size_t)c.m_tiles * c.n_tiles * 4;
}

template <int BN, int STAGES, bool SF_TMA>
w4a8_status launch(const CUtensorMap &tw, const uint8_t *xq, const Params &prm, const Cfg &c,
                   cudaStream_t stream)
{
    using L = Layout<BN, STAGES>;
    CUtensorMap tx, tsf;
    if (!tmap_bytes(&tx, xq, prm.M, prm.K, BN, 128)) return W4A8_ERR_CUDA;
    if (SF_TMA) {
        if (!tmap_bytes(&tsf, prm.we, prm.N, prm.K / 32, BM, 16, CU_TENSOR_MAP_SWIZZLE_NONE)) return W4A8_ERR_CUDA;
    } else {
        tsf = tx;  // unused
    }
    auto kern = mxfp4_tc_kernel<BN, STAGES, SF_TMA>;
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL) != cudaSuccess)
            return W4A8_ERR_CUDA;
        attr_done[dev] = 1;
    }
    dim3 grid(c.n_tiles, c.m_tiles, c.KS);
    kern<<<grid, NUM_THREADS, L::TOTAL, stream>>>(tw, tx, tsf, prm);
    return w4a8_launch_status();
}

}  // namespace tcg
}  // namespace w4a8

using namespace w4a8::tcg;

bool w4a8_tc_mxfp4_supported(const void *xq, const void *wp, const void *we, const void *out, int64_t M,
                             int64_t N, int64_t K)
{
    if (K % 128 != 0 || K < 128 || K > (1ll << 30) || M < 1 || M > (1ll << 30) || N < 1 || N > (1ll << 30))
        return false;
    if (!w4a8_aligned(wp, 32) || !w4a8_aligned(xq, 16) || !w4a8_aligned(we, 4) || !w4a8_aligned(out, 2))
        return false;
    const Cfg c = choose(M, N, K);
    return c.m_tiles <= 65535 && encode_fn() != nullptr;
}

size_t w4a8_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, int policy)
{
    if (policy == 1 || K % 128 != 0 || K < 128) return 0;
    return workspace_for(choose(M, N, K), M, N);
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
    prm.partials = nullptr;
    prm.counters = nullptr;
    prm.status = w4a8_device_status_ptr();
    if (!prm.status) return W4A8_ERR_CUDA;
    prm.M = (int)M;
    prm.N = (int)N;
    prm.K = (int)K;
    prm.KS = c.KS;
    prm.KT = (int)(K / BK);
    if (c.KS > 1) {
        size_t part = (size_t)c.KS * (size_t)M * (size_t)N * 4;
        part = (part + 255) / 256 * 256;
        prm.partials = static_cast<float *>(workspace);
        prm.counters = reinterpret_cast<int *>(static_cast<uint8_t *>(workspace) + part);
    }
    CUtensorMap tw;
    if (!tmap_w_fp4(&tw, wp, N, K)) return W4A8_ERR_CUDA;
    if (c.sf_tma && w4a8_aligned(we, 16)) {
        switch (c.BN) {
        case 16: return launch<16, 10, true>(tw, xq, prm, c, stream);
        case 32: return launch<32, 9, true>(tw, xq, prm, c, stream);
        case 64: return launch<64, 8, true>(tw, xq, prm, c, stream);
        case 128: return launch<128, 6, true>(tw, xq, prm, c, stream);
        default: return launch<256, 4, true>(tw, xq, prm, c, stream);
        }
    }
    switch (c.BN) {
    case 16: return launch<16, 10, false>(tw, xq, prm, c, stream);
    case 32: return launch<32, 9, false>(tw, xq, prm, c, stream);
    case 64: return launch<64, 8, false>(tw, xq, prm, c, stream);
    case 128: return launch<128, 6, false>(tw, xq, prm, c, stream);
    default: return launch<256, 4, false>(tw, xq, prm, c, stream);
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
