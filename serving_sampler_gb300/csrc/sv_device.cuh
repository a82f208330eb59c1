// Device-side building blocks of the specverify kernels (sm_103a):
// shared-memory barriers and bulk (TMA) copies written as inline PTX, bounded
// waits, packed bf16 maxima, Philox4x32-10 and the uniform used by every
// random draw.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "specverify.h"

namespace sv {

// Every wait on a barrier gives up after this many SM cycles (about two
// seconds at the boost clock); the kernel then records SV_ST_TIMEOUT instead
// of spinning forever.
constexpr long long kWaitLimitCycles = 4000000000LL;

// flags carried by per-row partial results
enum : uint32_t { kFlagNaN = 1u, kFlagTimeout = 2u, kFlagPosInf = 4u };

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// make initialised barriers visible to the async (bulk-copy) proxy
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// One probe of the barrier phase.  The hint lets the hardware suspend the
// thread (up to ~0.5 ms) until the phase completes instead of re-issuing.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(500000u)
        : "memory");
    return ok != 0;
}

// Wait for the given phase with a time limit (SM cycles).  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit = kWaitLimitCycles)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}

// ---- bulk copies (TMA, 1-D) ------------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// global -> shared copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned) that completes a transaction count on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// ---- programmatic dependent launch ----------------------------------------
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- packed bf16 / fp32 maxima that propagate NaN ---------------------------
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ float fmax_nan(float a, float b)
{
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}
// replace NaN halves of a bf16x2 word by -inf
__device__ __forceinline__ uint32_t bf16x2_nan_to_ninf(uint32_t w)
{
    uint32_t lo = w & 0xFFFFu, hi = w >> 16;
    if ((lo & 0x7FFFu) > 0x7F80u) lo = 0xFF80u;
    if ((hi & 0x7FFFu) > 0x7F80u) hi = 0xFF80u;
    return lo | (hi << 16);
}

// the two bf16 halves of a 32-bit word, widened exactly to fp32
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---- Philox4x32-10 (Salmon et al., SC'11) ----------------------------------
struct PhiloxKey {
    uint32_t k0, k1;
};

__device__ __forceinline__ PhiloxKey philox_key(uint64_t seed)
{
    return PhiloxKey{static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, PhiloxKey key)
{
    uint32_t k0 = key.k0, k1 = key.k1;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        // one 32 x 32 -> 64-bit product each: high and low halves from the same multiply
        const uint64_t pa = static_cast<uint64_t>(0xD2511F53u) * c.x;
        const uint64_t pb = static_cast<uint64_t>(0xCD9E8D57u) * c.z;
        c = make_uint4(static_cast<uint32_t>(pb >> 32) ^ c.y ^ k0, static_cast<uint32_t>(pb),
                       static_cast<uint32_t>(pa >> 32) ^ c.w ^ k1, static_cast<uint32_t>(pa));
    }
    return c;
}

// Uniform in (0, 1) from one 32-bit word: (2 * (w >> 9) + 1) * 2^-24.  The
// mantissa trick builds 1 + (w >> 9) * 2^-23 and subtracts 1 - 2^-24; both
// steps are exact in fp32.
__device__ __forceinline__ float uniform_from_word(uint32_t w)
{
    return __uint_as_float(0x3F800000u | (w >> 9)) - __uint_as_float(0x3F7FFFFFu);
}

// 1 - u for the same word, also exact: (2 * (2^23 - 1 - (w >> 9)) + 1) * 2^-24
__device__ __forceinline__ float one_minus_uniform_from_word(uint32_t w)
{
    return uniform_from_word(~w);
}

// counter layout of the library: (x >> 2, row, tag, 0), word x & 3
// uniform tags: the accept test, the residual race and the bonus race
enum : uint32_t { kTagAccept = 0, kTagResidual = 1, kTagBonus = 2 };

__device__ __forceinline__ uint4 philox_block(PhiloxKey key, uint32_t x4, uint32_t row, uint32_t tag)
{
    return philox4x32_10(make_uint4(x4, row, tag, 0u), key);
}

// ---- (value, index) argmax state --------------------------------------------
struct ArgMax {
    float v;    // best value seen (never NaN); -inf when nothing was seen
    int32_t i;  // its index; INT32_MAX when nothing beat -inf
};

__device__ __forceinline__ bool argmax_better(float v, int32_t i, const ArgMax& a)
{
    return v > a.v || (v == a.v && i < a.i);
}

// ---- shared-memory 16-bit accesses at 32-bit shared addresses, values in 32-bit registers ----
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr)
{
    uint32_t v;
    asm("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
// no memory clobber: callers order these stores against readers with a barrier
__device__ __forceinline__ void sts_u16(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "r"(v));
}

// ---- the temperature's scale of logits in log2 units ------------------------
// c = log2(e) / T for T > 0, held at or above 2^-100 so that T = +inf (every logit the same
// weight) still maps a -inf logit to -inf rather than to -inf * 0 = NaN; any finite logit of
// magnitude below 2^70 then scales to less than 2^-30 and weighs 1 in fp32, as at c = 0.
__device__ __forceinline__ float temp_scale(float T)
{
    return fmaxf(1.4426950408889634f / T, 0x1p-100f);
}

// ---- fp32 pairs, exponentials, loads and warp maxima shared by the kernels ----
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// two fp32 values in one 64-bit register, for the packed f32x2 instructions
__device__ __forceinline__ unsigned long long pack2(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(unsigned long long v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long sub2(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// the bf16x2 word w as two fp32 values (exact) in one 64-bit register
__device__ __forceinline__ unsigned long long bf16x2_to_f32x2(uint32_t w)
{
    return pack2(bf16_lo(w), bf16_hi(w));
}

// 16-byte read-only global load
__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// maximum over the warp (all lanes take part; no NaN among the inputs)
__device__ __forceinline__ float warp_max(float v)
{
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

}  // namespace sv
