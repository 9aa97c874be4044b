// tc_sched.cuh -- pieces shared by the tensor-core GEMM kernels: the data-parallel + stream-K
// work split, its unit arithmetic, and the bounded mbarrier waits that report a timeout in the
// library's device status block.
#pragma once
#include <stdint.h>

#include "tc_ptx.cuh"

namespace w4a8 {
namespace tcs {

constexpr int BM = 128;                       // weight rows per tile (MMA M)
constexpr long long WAIT_BUDGET = 1ll << 29;  // clock cycles (a quarter second or so)
constexpr long long DRAIN_BUDGET = 1ll << 24;

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

// First stream-K unit of CTA c, and the CTA that owns stream-K unit u, for the even split of RU
// units over the first G CTAs (RU >= G).
__device__ __forceinline__ long long unit_start(long long c, long long RU, int G) { return c * RU / G; }
__device__ __forceinline__ int unit_owner(long long u, long long RU, int G) { return (int)(((u + 1) * G - 1) / RU); }

// Work split (data-parallel + stream-K hybrid).  With T tiles of U units on G CTAs, every CTA
// owns D = T / G whole tiles (tiles R + c*D ... R + c*D + D - 1, R = T - D*G), and the first R
// tiles' RU = R*U units are split evenly over the first Gsk = min(G, RU) CTAs: CTA c < Gsk takes
// stream-K units [c*RU/Gsk, (c+1)*RU/Gsk) (at least one, so a split tile's contributors are
// consecutive CTAs), which touch tiles t_first..t_last; the first and last of those may be
// shared with neighbouring CTAs.
// Processing order: the two split stream-K tiles (the first and the last, where split) -- the one
// with fewer of this CTA's units first -- then the remaining stream-K tiles, then the whole
// data-parallel tiles.  The split tiles' fix-up (partial store, arrival count, last-arrival
// reduction) then runs in the epilogue while the MMAs of whole tiles proceed, and a CTA that owns
// whole tiles ends on a direct store.  Short split segment first: its partial is in long before the
// tile's other contributors finish, so the CTA is not that tile's last arrival; a long first
// segment ends with its neighbours' and often makes the CTA reduce that tile mid-way and then
// reduce its last tile too, two fix-ups in a row at the end of the kernel.
// a / b for a >= 0, b > 0: a 32-bit division when a fits (the common case), else 64-bit.
__device__ __forceinline__ long long div_nonneg(long long a, int b)
{
    return a <= 0x7fffffffLL ? (long long)((unsigned)a / (unsigned)b) : a / b;
}

struct Sched {
    long long u_begin, u_end, A, L;  // stream-K unit range, units of the split first / last tile
    long long A0;                    // units processed before the split last tile's (A or 0)
    int U, t_first, t_last, S_sk, S, dp_t0, D, n_sk, n_units;
    bool pf, pl, lf;                 // first / last stream-K tile split; lf: the last one goes first
    __device__ Sched(int cta, int Gsk, long long RU, int D_, int R, int U_) : U(U_), D(D_)
    {
        u_begin = cta < Gsk ? (long long)cta * RU / Gsk : RU;
        u_end = cta < Gsk ? (long long)(cta + 1) * RU / Gsk : RU;
        const long long ub = u_begin, ue = u_end;
        t_first = (int)(ub / U_);
        t_last = ue > ub ? (int)((ue - 1) / U_) : t_first - 1;
        S_sk = t_last - t_first + 1;
        pf = S_sk >= 1 && ((ub % U_) != 0 || (S_sk == 1 && ue - ub < U_));
        pl = S_sk >= 2 && (ue % U_) != 0;
        A = pf ? min(ue, (long long)(t_first + 1) * U_) - ub : 0;
        L = pl ? ue - (long long)t_last * U_ : 0;
        lf = pf && pl && L < A;
        A0 = lf ? 0 : A;
        dp_t0 = R + cta * D_;
        S = S_sk + D_;
        n_sk = (int)(ue - ub);
        n_units = n_sk + D_ * U_;
    }
    // global unit (tile * U + unit within the tile) processed at position p (0 <= p < n_units)
    __device__ long long unit_at(long long p) const
    {
        if (p < n_sk) {
            if (p < A0) return u_begin + p;
            if (p < A0 + L) return (long long)t_last * U + (p - A0);
            return u_begin + (p - L);
        }
        const unsigned q = (unsigned)(p - n_sk);  // < D * U: fits in 32 bits
        const unsigned qt = q / (unsigned)U;
        return (long long)(dp_t0 + (int)qt) * U + (long long)(q - qt * (unsigned)U);
    }
    // weight tile coordinates of the ring fill that starts at k-tile position i
    __device__ void fill_at(int i, int m_tiles, int &kt, int &n0) const
    {
        const long long u = unit_at(i / 4);
        const int t = (int)div_nonneg(u, U);
        kt = (int)(u - (long long)t * U) * 4 + (i & 3);
        n0 = (int)((unsigned)t / (unsigned)m_tiles) * BM;
    }
    // the same, plus the token tile index of k-tile i's tile
    __device__ void fill_at(int i, int m_tiles, int &kt, int &n0, int &mt) const
    {
        const long long u = unit_at(i / 4);
        const int t = (int)div_nonneg(u, U);
        kt = (int)(u - (long long)t * U) * 4 + (i & 3);
        n0 = (int)((unsigned)t / (unsigned)m_tiles) * BM;
        mt = (int)((unsigned)t % (unsigned)m_tiles);
    }
    // tile of the k-th segment in processing order, and its unit range [a, b)
    __device__ int seg_tile(int k) const
    {
        if (k >= S_sk) return dp_t0 + (k - S_sk);
        int s = k;
        if (pl) s = (pf && !lf) ? (k == 0 ? 0 : (k == 1 ? S_sk - 1 : k - 1)) : (k == 0 ? S_sk - 1 : k - 1);
        return t_first + s;
    }
    __device__ void seg_units(int k, long long &a, long long &b) const
    {
        const long long t = seg_tile(k);
        if (k >= S_sk) {
            a = t * U;
            b = a + U;
            return;
        }
        a = max(u_begin, t * U);
        b = min(u_end, (t + 1) * U);
    }
};

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

// Host side: the work split for T tiles of U units on at most n_sms CTAs.
struct SkSplit {
    int G, D, R, Gsk;
    long long RU;
};
inline SkSplit sk_split(long long T, int U, int n_sms)
{
    SkSplit k;
    const long long TU = T * U;
    k.G = (int)(TU < n_sms ? TU : n_sms);
    k.D = (int)(T / k.G);  // whole tiles per CTA
    k.R = (int)(T - (long long)k.D * k.G);  // tiles split stream-K over the first Gsk CTAs
    k.RU = (long long)k.R * U;
    k.Gsk = (int)(k.RU < 1 ? 1 : (k.RU < k.G ? k.RU : k.G));
    return k;
}

}  // namespace tcs
}  // namespace w4a8
