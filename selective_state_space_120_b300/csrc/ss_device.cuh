// Device-side building blocks of the selective-scan kernels (sm_103a).
//
// Math follows "Mamba Series from Selective State Spaces to Visual State Space
// Models", section "mathematical form of the selective SSM":
//   Abar = exp(Delta*A), Bbar*u = Delta*B*u, Delta = softplus(raw + bias),
// and the Mamba block's SiLU gate.  Exponentials run on the SFU as base-2
// exponentials: A is pre-scaled by log2(e) once per channel, so
// exp(Delta*A) = ex2(Delta * A*log2(e)).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace ssk {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr unsigned kFull = 0xffffffffu;

// Status word of the library on each device: bit 0 = a bounded wait gave up.
// (All kernels live in one translation unit, which includes this header once.)
__device__ unsigned int g_status = 0;
// Time budget (ns) of every bounded wait; 1 s unless changed for diagnostics.
__device__ unsigned long long g_wait_budget_ns = 1000000000ull;
// Diagnostics only (0 in normal use).  Bit 0: the first CTA of each TMA scan
// launch never issues the copies of its first tile, so its wait for that tile
// runs out after the wait budget -- the way the timeout path is tested.
__device__ unsigned int g_debug_flags = 0;

// ------------------------------------------------------------------ SFU math
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(x) = ln(1 + e^x).  With e = 2^(x*log2 e):
//   e < 1/32 : the Taylor series ln(1+e) = e - e^2/2 + e^3/3 - e^4/4
//              (dropped terms below e^5/5, i.e. relative error < 2e-7), which
//              keeps full relative accuracy for tiny Delta where ln(1+e)
//              computed through 1+e would lose it;
//   otherwise: ln2 * log2(1 + e);
//   x > 15   : x itself (the two differ by less than 3.1e-7 relative).
// softplus_from_exp takes e = 2^(x*log2 e) computed by the caller.
__device__ __forceinline__ float softplus_from_exp(float x, float e) {
    const float series = e * fmaf(e, fmaf(e, fmaf(e, -0.25f, 0.333333343f), -0.5f), 1.0f);
    const float via_log = kLn2 * lg2(1.0f + e);
    const float r = (e < 0.03125f) ? series : via_log;
    return (x > 15.0f) ? x : r;
}
__device__ __forceinline__ float softplus(float x) { return softplus_from_exp(x, ex2(x * kLog2e)); }

// SiLU(z) = z * sigmoid(z) = z / (1 + e^-z).  For z -> -inf the exponential
// overflows to +inf, the reciprocal to 0 and the result to -0.
__device__ __forceinline__ float silu(float z) { return z * rcp(1.0f + ex2(-z * kLog2e)); }

// ------------------------------------------------------------------ I/O types
template <typename IO> struct IOT;
// Prefetch loads as volatile asm: the compiler keeps them where they are
// written (before the barrier and scan that hide their latency) instead of
// sinking them to their first use.
__device__ __forceinline__ unsigned short ld_pref_u16(const void *p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_pref_f32(const void *p) {
    float v;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float4 ld_pref_v4(const void *p) {
    float4 v;
    asm volatile("ld.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// load_raw / widen split a load from its conversion, so a prefetched value can
// stay in flight until it is used.
template <> struct IOT<float> {
    using Raw = float;
    static __device__ __forceinline__ float from_f(float v) { return v; }
    static __device__ __forceinline__ float load(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ Raw load_raw(const float *p) { return ld_pref_f32(p); }
    static __device__ __forceinline__ float widen(Raw r) { return r; }
};
template <> struct IOT<__nv_bfloat16> {
    using Raw = unsigned short;
    static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
        const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(p));
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
    static __device__ __forceinline__ Raw load_raw(const __nv_bfloat16 *p) {
        return ld_pref_u16(p);
    }
    static __device__ __forceinline__ float widen(Raw r) {
        return __uint_as_float(static_cast<uint32_t>(r) << 16);
    }
};

// Two floats -> one 32-bit word of two bf16 (round to nearest even), low half first.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Unpacks a 32-bit word of the I/O type into floats (2 bf16 values or 1 float).
__device__ __forceinline__ void unpack_word(uint32_t w, float *dst, __nv_bfloat16 *) {
    dst[0] = __uint_as_float(w << 16);
    dst[1] = __uint_as_float(w & 0xffff0000u);
}
__device__ __forceinline__ void unpack_word(uint32_t w, float *dst, float *) {
    dst[0] = __uint_as_float(w);
}

// ------------------------------------------------------------------ smem tiles
// Raw tiles are written by TMA with 64-byte rows and the 64-byte swizzle:
// address bits [7:8] are XORed into bits [4:5] (16-byte chunk index).  Tiles
// start on 1024-byte boundaries, so offsets within a tile can be swizzled alone.
__device__ __forceinline__ int swz64(int off) { return off ^ (((off >> 7) & 3) << 4); }

// Step-pair slots of the prepared (Delta', x) and (gate, D*u*gate) rows are
// XOR-swizzled inside groups of eight 16-byte slots so that the prep lanes,
// which each own a run of consecutive slots, store with few bank conflicts.
__device__ __forceinline__ int swz_slot(int tp) { return tp ^ ((tp >> 3) & 7); }

// Reads E consecutive I/O elements of row `row` of a swizzled 64-byte-row tile,
// starting at column col0, widened to float.
template <typename IO, int E>
__device__ __forceinline__ void load_tile_row(const uint8_t *tile, int row, int col0, float *v) {
    constexpr int ES = sizeof(IO);
    constexpr int BYTES = E * ES;
    constexpr int PER = 4 / ES;  // elements per 32-bit word
    const int off = row * 64 + col0 * ES;
    if constexpr (BYTES >= 16) {
#pragma unroll
        for (int c = 0; c < BYTES / 16; ++c) {
            const uint4 w = *reinterpret_cast<const uint4 *>(tile + swz64(off + 16 * c));
            float *d = v + (16 / ES) * c;
            unpack_word(w.x, d + 0 * PER, (IO *)nullptr);
            unpack_word(w.y, d + 1 * PER, (IO *)nullptr);
            unpack_word(w.z, d + 2 * PER, (IO *)nullptr);
            unpack_word(w.w, d + 3 * PER, (IO *)nullptr);
        }
    } else if constexpr (BYTES == 8) {
        const uint2 w = *reinterpret_cast<const uint2 *>(tile + swz64(off));
        unpack_word(w.x, v, (IO *)nullptr);
        unpack_word(w.y, v + PER, (IO *)nullptr);
    } else {
        static_assert(BYTES == 4, "prep lanes read at least one 32-bit word");
        const uint32_t w = *reinterpret_cast<const uint32_t *>(tile + swz64(off));
        unpack_word(w, v, (IO *)nullptr);
    }
}

// ------------------------------------------------------------------ mbarrier / TMA
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for the phase with the given parity to complete, for at most `budget`
// nanoseconds.  Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t budget) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > budget) return false;
    }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void report_timeout() { atomicOr(&g_status, 1u); }

// ------------------------------------------------------------------ traversal orders
// Division by a runtime-invariant divisor through a multiply-high (Granlund and
// Montgomery, "Division by Invariant Integers using Multiplication", 1994):
// for 1 <= d < 2^31 and 0 <= n < 2^31, n / d = (mulhi(m, n) + n) >> l with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1.
struct FastDiv {
    uint32_t d, m, l;
    __host__ __device__ FastDiv() : d(1), m(1), l(0) {}
    __host__ explicit FastDiv(uint32_t dv) : d(dv) {
        l = 0;
        while ((1ull << l) < dv) ++l;
        m = (uint32_t)((((1ull << l) - dv) << 32) / dv + 1);
    }
    __device__ __forceinline__ uint32_t div(uint32_t n) const {
        return (uint32_t)(((uint64_t)__umulhi(m, n) + n) >> l);
    }
};

// Position (row-major index on the H x W map; a plain sequence is H = 1) that
// scan step s of a direction with the given order visits:
//   0 row-major, 1 column-major (the transposed map), 2 and 3 their reverses.
__device__ __forceinline__ int64_t position_of(int order, int64_t s, int64_t L, int H, int W,
                                               const FastDiv &divH) {
    if (order == 2 || order == 3) s = L - 1 - s;  // reversed orders
    if (order == 1 || order == 3) {               // column-major
        const uint32_t q = divH.div((uint32_t)s);
        const uint32_t r = (uint32_t)s - q * (uint32_t)H;
        return (int64_t)r * W + q;
    }
    return s;
}

// Windowed traversals ("LocalMamba: Visual State Space Model with Windowed
// Selective Scan": the map is divided into windows and scanned window by
// window).  The Hm x Wm map is cut into w x w windows -- those of the last band
// of rows and of the last column cut short -- visited row-major, each window
// row-major.  The column-major variant is the same walk on the transposed map.
// WinWalk steps through it one cell at a time, forward or backward, without
// divisions; seek() places it at a step.
struct WinWalk {
    int Hm, Wm, w;
    int band, j, rr, cc;  // band of rows (band*w ..), window in the band, cell in the window
    __device__ __forceinline__ int hb() const { return min(w, Hm - band * w); }
    __device__ __forceinline__ int wj() const { return min(w, Wm - j * w); }
    __device__ __forceinline__ void seek(uint32_t s) {
        const uint64_t bandsz = (uint64_t)w * (uint64_t)Wm;  // cells of a full band
        band = (int)(s / bandsz);
        uint32_t rem = (uint32_t)(s - (uint64_t)band * bandsz);
        const int h = hb();
        j = (int)(rem / (uint32_t)(h * w));
        rem -= (uint32_t)(j * h * w);
        const int ww = wj();
        rr = (int)(rem / (uint32_t)ww);
        cc = (int)rem - rr * ww;
    }
    __device__ __forceinline__ void next() {
        if (++cc < wj()) return;
        cc = 0;
        if (++rr < hb()) return;
        rr = 0;
        if (++j * w < Wm) return;
        j = 0;
        ++band;
    }
    __device__ __forceinline__ void prev() {
        if (--cc >= 0) return;
        if (--rr >= 0) {
            cc = wj() - 1;
            return;
        }
        if (--j >= 0) {
            rr = hb() - 1;
            cc = wj() - 1;
            return;
        }
        --band;
        j = (Wm - 1) / w;
        rr = hb() - 1;
        cc = wj() - 1;
    }
    __device__ __forceinline__ int row() const { return band * w + rr; }
    __device__ __forceinline__ int col() const { return j * w + cc; }
};

// Step of the windowed walk over an Hm x Wm map at which cell (r, c) is visited.
__device__ __forceinline__ uint32_t win_step(int r, int c, int Hm, int Wm, int w) {
    const int band = r / w, rr = r - band * w, j = c / w, cc = c - j * w;
    const int hb = min(w, Hm - band * w), wj = min(w, Wm - j * w);
    // band * w * Wm and j * hb * w count cells before this one: below H*W < 2^31
    return (uint32_t)((int64_t)band * w * Wm + (int64_t)j * hb * w + rr * wj + cc);
}

// Traversal codes beyond the four of SS2D (match SS_DIR_* of the C ABI).
enum { ORD_K_WIN = 4, ORD_K_WIN_COL = 5, ORD_K_WIN_REV = 6, ORD_K_WIN_COL_REV = 7 };

// Step at which a direction with the given order visits cell (r, c) of the
// H x W map: the inverse of the traversal.
__device__ __forceinline__ uint32_t step_of(int order, int r, int c, int H, int W, int w) {
    const uint32_t L = (uint32_t)H * (uint32_t)W;
    uint32_t s;
    switch (order) {
    case 0: return (uint32_t)(r * W + c);
    case 1: return (uint32_t)(c * H + r);
    case 2: return L - 1 - (uint32_t)(r * W + c);
    case 3: return L - 1 - (uint32_t)(c * H + r);
    case ORD_K_WIN: return win_step(r, c, H, W, w);
    case ORD_K_WIN_COL: return win_step(c, r, W, H, w);
    case ORD_K_WIN_REV: s = win_step(r, c, H, W, w); return L - 1 - s;
    default: s = win_step(c, r, W, H, w); return L - 1 - s;
    }
}

// Positions of consecutive scan steps of a direction with a column order (1, 3)
// or a windowed one (4..7), one step at a time: start() places it at step s (a
// step past the end is treated as the last), pos_next() returns the position of
// the current step and moves to the next.
struct OrderWalk {
    int order, H, W;
    int r, c;    // column orders: cell of the current step
    WinWalk ww;  // windowed orders
    __device__ __forceinline__ void start(int ord, int H_, int W_, int win, int64_t L, int64_t s) {
        order = ord;
        H = H_;
        W = W_;
        const int64_t sc = s < L ? s : L - 1;
        if (order == 1 || order == 3) {
            const uint32_t cm = (uint32_t)(order == 3 ? L - 1 - sc : sc);  // column-major index
            c = (int)(cm / (uint32_t)H);
            r = (int)(cm - (uint32_t)c * (uint32_t)H);
        } else {
            const bool tr = order == ORD_K_WIN_COL || order == ORD_K_WIN_COL_REV;
            ww.Hm = tr ? W : H;
            ww.Wm = tr ? H : W;
            ww.w = win;
            ww.seek((uint32_t)(order >= ORD_K_WIN_REV ? L - 1 - sc : sc));
        }
    }
    __device__ __forceinline__ int64_t pos_next() {
        int64_t p;
        if (order == 1 || order == 3) {
            p = (int64_t)r * W + c;
            if (order == 1) {
                if (++r == H) {
                    r = 0;
                    ++c;
                }
            } else if (--r < 0) {
                r = H - 1;
                --c;
            }
        } else {
            const bool tr = order == ORD_K_WIN_COL || order == ORD_K_WIN_COL_REV;
            p = tr ? (int64_t)ww.col() * W + ww.row() : (int64_t)ww.row() * W + ww.col();
            if (order >= ORD_K_WIN_REV) ww.prev();
            else ww.next();
        }
        return p;
    }
};

// ------------------------------------------------------------------ lane-group reduction
// R lanes (R a power of two) each hold R partial sums v[0..R): one
// per step of an R-step block.  Afterwards the lane with group index g holds the
// sum over the R lanes of v[g].  log2(R) butterfly rounds; each round halves the
// values a lane keeps and exchanges the other half with its partner.
// The R lanes of a group sit LSTRIDE lanes apart (lane = g * LSTRIDE + q).
template <int R, int LSTRIDE = 1>
__device__ __forceinline__ float transpose_reduce(float (&v)[R], int g) {
    if constexpr (R == 1) {
        return v[0];
    } else {
#pragma unroll
        for (int m = R / 2; m >= 1; m >>= 1) {
            const bool up = (g & m) != 0;
#pragma unroll
            for (int i = 0; i < m; ++i) {
                const float send = up ? v[i] : v[i + m];
                const float keep = up ? v[i + m] : v[i];
                v[i] = keep + __shfl_xor_sync(kFull, send, m * LSTRIDE);
            }
        }
        return v[0];
    }
}

}  // namespace ssk
