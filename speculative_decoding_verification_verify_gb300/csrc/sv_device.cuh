// sv_device.cuh -- device-side building blocks of the verifier kernels (sm_103a).
//
// Everything here is written for the GPU path only; the CPU oracle has its own code.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sv_check.cuh"

namespace sv {

constexpr int NT = 256;       // threads per CTA of the finalising, residual and block kernels
constexpr int NW = NT / 32;   // their warps
constexpr int NT_S = 768;     // threads of a streaming CTA (one CTA per SM)
#ifndef SV_NT_SV
#define SV_NT_SV 512
#endif
// The variant streaming kernels (a temperature per request, top-k / top-p) hold both folds'
// state: fewer warps per CTA leave each thread the registers to do so without spilling.
constexpr int NT_SV = SV_NT_SV;
#ifndef SV_NT_S4
#define SV_NT_S4 640
#endif
constexpr int NT_S4 = SV_NT_S4;  // the filtered one-temperature kind: 20 warps keep its fold in registers
__host__ __device__ constexpr int stream_threads(int kind)
{
    return kind == 2 || kind == 3 ? NT_SV : (kind == 4 ? NT_S4 : NT_S);
}
#ifndef SV_RESID_GROUPS
#define SV_RESID_GROUPS 2
#endif
constexpr int RESID_GROUPS = SV_RESID_GROUPS;  // 8-column groups a lane of the residual sums loads at once
constexpr int MAX_RPR = 64;   // rows per request: k + 1 <= 64 (chain) or N <= 64 (tree)
constexpr int B_MAX = 65536;  // most requests per call (size of the fixed counter region)
constexpr int C2_MAX = 1024;  // upper bound on column chunks of the residual kernel
#ifndef SV_CHUNK_VEC
#define SV_CHUNK_VEC 512
#endif
constexpr int CHUNK_VEC = SV_CHUNK_VEC;  // 16-byte vectors per streaming chunk (one record each)
constexpr float NEG_INF = -__builtin_huge_valf();
constexpr float POS_INF = __builtin_huge_valf();

// ---------------------------------------------------------------------------------------------
// Kernel parameters (one struct, passed by value).
// ---------------------------------------------------------------------------------------------
struct Params {
    const void *logits;          // [B][rpr][V]
    const int32_t *drafts;       // chain: [B][k]
    const float *q;              // chain: [B][k][V] draft distributions, or null (one-hot)
    const int32_t *node_tokens;  // tree: [B][N]
    const int32_t *parents;      // tree: [B][N]
    int B, k, rpr, is_tree;
    int block;                   // chains: block verification instead of token-by-token
    int64_t V;
    float cs;                    // log2(e) / T: p is proportional to 2^(logit * cs)
    const float *temps;          // [B] per-request temperatures (0: greedy request), or null
    const int32_t *top_k;        // [B] per-request top-k (<= 0 or >= V: off), or null
    const float *top_p;          // [B] per-request top-p (>= 1: off), or null
    float *thr;                  // [B * rpr] logit threshold of each row (-inf: not filtered)
    float thr_single, thr_acc;   // relaxed thresholds of target-only decisions (1: exact)
    uint32_t key0, key1, off0, off1;
    int64_t total;               // B * rpr * V
    int64_t nch;                 // streaming chunks per row
    int64_t nchunks;             // B * rpr * nch
    int64_t cpc;                 // chunks per streaming CTA
    int G;                       // streaming CTAs
    int mis;                     // logits base address mod 16, in elements
    int32_t *out_tokens;         // chain [B][k+1], tree [B][N]
    int32_t *accept_len;         // [B]
    int32_t *accept_index;       // tree [B][N]
    float *out_probs;            // chain [B][k+1][3] or null
    int32_t *dev_status;         // or null
    // workspace
    unsigned *cnt2;              // [B] arrivals at the residual kernel's counter
    float4 *recs;                // [B * rpr * nch] one record per streaming chunk
    float *caps;                 // [B * rpr] logit of node j's token in its parent's row
    int4 *pend;                  // [B] residual draw pending: {row, mc bits, total bits, flag}
    float2 *recs2;               // [B * C2 * NW] residual-kernel records
    float4 *bpend;               // block with q: [B * rpr] per row {max ref, total, prefix weight, 1}
    float2 *recs3;               // block with q: [B * rpr * C2 * NW] per (row, chunk, warp) sums
    int C2;                      // residual-kernel column chunks per request
    int64_t Ec2;                 // columns per residual chunk
};

// ---------------------------------------------------------------------------------------------
// PTX helpers.
// ---------------------------------------------------------------------------------------------
// 16-byte streaming load through the non-coherent path, not kept in L1.
__device__ __forceinline__ uint4 ldg_stream(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// The same with L2 priority evict-first: a line this load brings into L2 is among the first to
// go, so that the lines a previous pass left there at normal priority stay.
__device__ __forceinline__ uint4 ldg_stream_ef(const void *p)
{
    uint4 r;
    unsigned long long pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p), "l"(pol));
    return r;
}

// 2^x on the SFU (approximate, flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max that returns NaN when either input is NaN.
__device__ __forceinline__ float fmax_nan(float a, float b)
{
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Programmatic dependent launch: the finalising kernel may start while the streaming kernel
// runs; it reads only inputs until pdl_wait(), which returns once the streaming grid has
// completed and its writes are visible.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 16-byte asynchronous copy global -> shared (both addresses 16-byte aligned), in the thread's
// current cp.async group.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gsrc)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ void raise_status(int32_t *st, int code)
{
    if (st && code) atomicMax(st, code);
}

// ---------------------------------------------------------------------------------------------
// Element access per dtype: VEC elements per 16-byte vector.
// ---------------------------------------------------------------------------------------------
template <typename T>
struct Elt;

template <>
struct Elt<__nv_bfloat16> {
    static constexpr int VEC = 8;
    static __device__ __forceinline__ float load(const void *row, int64_t c)
    {
        return __uint_as_float((uint32_t)__ldg((const unsigned short *)row + c) << 16);
    }
    static __device__ __forceinline__ void unpack(const uint4 &w, float (&x)[VEC])
    {
        x[0] = bf_lo(w.x); x[1] = bf_hi(w.x);
        x[2] = bf_lo(w.y); x[3] = bf_hi(w.y);
        x[4] = bf_lo(w.z); x[5] = bf_hi(w.z);
        x[6] = bf_lo(w.w); x[7] = bf_hi(w.w);
    }
    static __device__ __forceinline__ float vmax(const uint4 &w)
    {
        uint32_t m = bmax2_nan(bmax2_nan(w.x, w.y), bmax2_nan(w.z, w.w));
        return fmax_nan(bf_lo(m), bf_hi(m));
    }
};

template <>
struct Elt<float> {
    static constexpr int VEC = 4;
    static __device__ __forceinline__ float load(const void *row, int64_t c)
    {
        return __ldg((const float *)row + c);
    }
    static __device__ __forceinline__ void unpack(const uint4 &w, float (&x)[VEC])
    {
        x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
    }
    static __device__ __forceinline__ float vmax(const uint4 &w)
    {
        return fmax_nan(fmax_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                        fmax_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
};

// ---------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): counter (slot, request, off0, off1),
// key (key0, key1).  u = word 0, v = word 1, each mapped to (x >> 8) * 2^-24.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0;
        const uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return make_uint4(c0, c1, c2, c3);
}

// log2(e) / T in double, rounded once: the scale of a request's logits (T > 0).
__device__ __forceinline__ float cs_of(float T) { return (float)(1.4426950408889634 / (double)T); }

__device__ __forceinline__ float u01(uint32_t x) { return (float)(x >> 8) * 5.9604644775390625e-08f; }

__device__ __forceinline__ float2 uniforms(const Params &P, uint32_t slot, uint32_t req)
{
    const uint4 w = philox4x32_10(slot, req, P.off0, P.off1, P.key0, P.key1);
    return make_float2(u01(w.x), u01(w.y));
}

// ---------------------------------------------------------------------------------------------
// Online (max, sum) records: a record (mc, s) stands for s * 2^mc in the scaled domain.  A
// record that has seen no finite logit has s = 0 (or NaN when it saw a NaN); its reference mc
// is never used then, so merges test s, not mc.
// ---------------------------------------------------------------------------------------------
constexpr float REF_NONE = -3.4028234663852886e38f;  // reference before any finite logit

__device__ __forceinline__ void rec_merge(float &mc, float &s, float omc, float os)
{
    const float nm = fmaxf(mc, omc);
    const float a = (s == 0.f) ? 0.f : s * ex2(mc - nm);
    const float b = (os == 0.f) ? 0.f : os * ex2(omc - nm);
    mc = nm;
    s = a + b;
}

// Merge the warp's records into one, in every lane: the largest reference first, then each
// lane's sum rescaled to it once and a plain warp sum.  A record with s = 0 has the reference
// REF_NONE (a lane that saw a finite logit has a term 2^0 = 1 in its sum), so it cannot raise the
// reference; a NaN sum, or a +inf logit (reference +inf, rescale 2^NaN), makes the result NaN.
__device__ __forceinline__ void warp_rec_merge(float &mc, float &s)
{
    float M = mc;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float v = (s == 0.f) ? 0.f : s * ex2(mc - M);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    mc = M;
    s = v;
}

// Argmax records: larger value wins, lower index on ties, NaN is sticky.
__device__ __forceinline__ void arg_merge(float &v, int &i, float ov, int oi)
{
    const bool nan_a = (v != v), nan_b = (ov != ov);
    if (nan_a || nan_b) {
        if (!nan_a) {
            v = ov;
            i = oi;
        }
        return;
    }
    if (ov > v || (ov == v && oi < i)) {
        v = ov;
        i = oi;
    }
}

__device__ __forceinline__ void warp_arg_merge(float &v, int &i)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, off);
        const int oi = __shfl_xor_sync(0xffffffffu, i, off);
        arg_merge(v, i, ov, oi);
    }
}

// ---------------------------------------------------------------------------------------------
// Geometry of the streaming chunks.  Row r is cut into nch chunks of CE = CHUNK_VEC * VEC
// columns whose boundaries fall on the flat array's 16-byte grid: chunk j covers columns
// [A + j * CE, A + (j + 1) * CE) of [0, V), A = -((r * V + mis) mod VEC) <= 0, so only a row's first
// chunk has an unaligned head and only its last an unaligned tail; nch = ceil((V + VEC - 1) / CE)
// covers every A, and a chunk past the row's end is empty.  The record of chunk (r, j) is
// r * nch + j, so a row's records are contiguous.  The streaming CTAs take equal runs of the
// B * rpr * nch chunks in that order.
// ---------------------------------------------------------------------------------------------
struct Seg {
    int64_t c0, c1;  // chunk columns [c0, c1)
    int64_t b0, b1;  // its vector body [b0, b1), 16-byte aligned
};

template <int VEC>
__device__ __forceinline__ Seg chunk_of(const Params &P, int64_t r, int64_t j)
{
    constexpr int64_t CE = (int64_t)CHUNK_VEC * VEC;
    const int64_t rowf = r * P.V;
    const int64_t A = -((rowf + P.mis) % VEC);
    int64_t p0 = A + j * CE, p1 = p0 + CE;
    if (p0 < 0) p0 = 0;
    if (p1 > P.V) p1 = P.V;
    if (p0 > p1) p0 = p1;
    int64_t a0 = p0 + (VEC - (rowf + p0 + P.mis) % VEC) % VEC;
    if (a0 > p1) a0 = p1;
    int64_t a1 = p1 - (rowf + p1 + P.mis) % VEC;
    if (a1 < a0) a1 = a0;
    Seg s;
    s.c0 = p0;
    s.c1 = p1;
    s.b0 = a0;
    s.b1 = a1;
    return s;
}

// Node relations: the chain is a path tree (node j >= 1 has parent j - 1 and token
// drafts[j - 1]); trees read parents / node_tokens.
__device__ __forceinline__ int node_parent(const Params &P, int b, int n)
{
    if (!P.is_tree) return n - 1;
    const int64_t i = (int64_t)b * P.rpr + n;
    return SV_INB(i, (int64_t)P.B * P.rpr, 101) ? __ldg(P.parents + i) : -1;
}

__device__ __forceinline__ int node_token(const Params &P, int b, int n)
{
    if (!P.is_tree) {
        const int64_t i = (int64_t)b * P.k + (n - 1);
        return SV_INB(i, (int64_t)P.B * P.k, 102) ? __ldg(P.drafts + i) : -1;
    }
    const int64_t i = (int64_t)b * P.rpr + n;
    return SV_INB(i, (int64_t)P.B * P.rpr, 103) ? __ldg(P.node_tokens + i) : -1;
}

}  // namespace sv
