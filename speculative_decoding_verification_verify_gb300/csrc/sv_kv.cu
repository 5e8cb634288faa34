// sv_kv.cu -- after tree verification, move each request's accepted-path KV rows to contiguous
// positions after its committed prefix and advance the committed length ("投机解码", section
// 与调度、KV 的交互, SGLang part: the committed length grows by the accepted count, and with
// topk > 1 the accepted path, which is not contiguous in the tree, is moved to contiguous
// positions; "Draft sources: draft models, n-gram, suffix decoding", section "SGLang's suffix
// automaton, in tree", the NGRAM decode-step walk-through: verification, then
// move_accept_tokens_to_target_kvcache).
//
// A copy of a few MB per call, so besides bandwidth its time is the chain of dependent memory
// round trips.  The KV cache is `planes` planes (one per layer and K or V), each
// [num_slots][row_bytes]; a request's work is planes x row_vec 16-byte vectors, K per thread
// (columns NT apart), CTAs over (chunk of NT*K vectors, request).  The prologue takes two round
// trips: the accepted path and committed length together, then the slots of the request's N tree
// positions (they depend on the committed length only).  A thread then loads its K vectors of up
// to SB path steps' source rows at once and stores them all, one round trip per SB steps.  That
// equals copying the steps one by one in path order as long as no step reads a slot an earlier
// step wrote; on a root-to-node path with distinct slots it never does (the source positions
// committed + a_i lie past every earlier destination committed + j, j < i, since a_i >= i).  When
// it does, the CTA copies step by step.  A column's steps stay with one thread, so a step that
// overwrites a row an earlier step read still comes after that read.
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"
#include "sv_check.cuh"

namespace svkv {

#ifndef SV_KV_NT
#define SV_KV_NT 128
#endif
#ifndef SV_KV_K
#define SV_KV_K 4
#endif
#ifndef SV_KV_SB
#define SV_KV_SB 2
#endif
#ifndef SV_KV_MINB
#define SV_KV_MINB 8
#endif
constexpr int NT = SV_KV_NT;    // threads per CTA
constexpr int K = SV_KV_K;      // 16-byte vectors (columns) per thread
constexpr int SB = SV_KV_SB;    // path steps whose rows a thread holds at once
// CTAs resident per SM the registers are budgeted for: most of a call's time is each CTA's chain
// of dependent round trips (indices, slots, data), so more CTAs in flight per SM hide more of it
// (two steps held and eight CTAs of 128 threads, 64 registers, beat four steps and five CTAs).
constexpr int CHUNK = NT * K;   // vectors per CTA
constexpr int MAX_NODES = 64;

// pool_vec: the pool's extent in 16-byte vectors (for the range checks of debug builds).
__global__ void __launch_bounds__(NT, SV_KV_MINB) kv_compact_kernel(uint4 *pool, int64_t num_slots, int64_t row_vec,
                                                        int64_t plane_vec, int64_t work, int64_t pool_vec,
                                                        const int32_t *slot_table, int max_pos,
                                                        const int32_t *committed_in, int32_t *committed_out,
                                                        const int32_t *accept_index, const int32_t *accept_len,
                                                        int N, int32_t *dev_status)
{
    __shared__ int64_t src_s[MAX_NODES], dst_s[MAX_NODES];
    __shared__ int32_t slot_s[MAX_NODES];
    // bit 0: a position error; bit 1: a slot error; bit 2: a step reads a slot an earlier step wrote
    __shared__ int flags;
    const int b = blockIdx.y, tid = threadIdx.x;
    // The three index reads are independent: one round trip.
    const int L = accept_len[b];
    const int c = committed_in[b];
    const int a = tid < N && SV_INB((int64_t)b * N + tid, (int64_t)gridDim.y * N, 801) ? accept_index[(int64_t)b * N + tid]
                                                                                  : 0;
    const bool first = blockIdx.x == 0 && tid == 0;
    if (L < 0) {  // a request the verifier faulted: nothing moves, nothing is committed
        if (first) committed_out[b] = c;
        return;
    }
    const bool pos_ok = c >= 0 && (int64_t)c + N <= max_pos && L < N;
    if (pos_ok && tid < N && SV_INB((int64_t)b * max_pos + c + tid, (int64_t)gridDim.y * max_pos, 802))
        slot_s[tid] = slot_table[(int64_t)b * max_pos + c + tid];
    if (tid == 0) flags = pos_ok ? 0 : 1;
    __syncthreads();
    if (pos_ok && tid <= L) {
        if (a < 0 || a >= N) {
            atomicOr(&flags, 1);
        } else {
            const int64_t s = slot_s[a], d = slot_s[tid];
            if (s < 0 || s >= num_slots || d < 0 || d >= num_slots) atomicOr(&flags, 2);
            src_s[tid] = s * row_vec;
            dst_s[tid] = d * row_vec;
        }
    }
    __syncthreads();
    const int err = flags & 3;
    if (err) {  // a position error outranks a slot error, as in a check of positions first
        if (first) {
            committed_out[b] = c;
            if (dev_status)
                atomicMax(dev_status, (err & 1) ? SPEC_VERIFY_DEV_BAD_KV_POSITION : SPEC_VERIFY_DEV_BAD_KV_SLOT);
        }
        return;
    }
    if (tid >= 2 && tid <= L) {
        const int64_t s = src_s[tid];
        for (int j = 1; j < tid; ++j)
            if (s == dst_s[j]) {
                atomicOr(&flags, 4);
                break;
            }
    }
    __syncthreads();
    const bool in_order = flags & 4;
    int64_t off[K];
    bool has[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int64_t e = (int64_t)blockIdx.x * CHUNK + tid + (int64_t)k * NT;
        const int64_t p = e / row_vec;
        off[k] = p * plane_vec + (e - p * row_vec);
        has[k] = e < work;
    }
    if (!in_order) {
        for (int i0 = 1; i0 <= L; i0 += SB) {
            uint4 v[SB][K];
#pragma unroll
            for (int u = 0; u < SB; ++u) {
                const int i = i0 + u;
                if (i <= L && src_s[i] != dst_s[i]) {
#pragma unroll
                    for (int k = 0; k < K; ++k)
                        if (has[k] && SV_INB(src_s[i] + off[k], pool_vec, 803)) v[u][k] = pool[src_s[i] + off[k]];
                }
            }
#pragma unroll
            for (int u = 0; u < SB; ++u) {
                const int i = i0 + u;
                if (i <= L && src_s[i] != dst_s[i]) {
#pragma unroll
                    for (int k = 0; k < K; ++k)
                        if (has[k] && SV_INB(dst_s[i] + off[k], pool_vec, 804)) pool[dst_s[i] + off[k]] = v[u][k];
                }
            }
        }
    } else {
        for (int i = 1; i <= L; ++i) {
            if (src_s[i] == dst_s[i]) continue;
            uint4 v[K];
#pragma unroll
            for (int k = 0; k < K; ++k)
                if (has[k] && SV_INB(src_s[i] + off[k], pool_vec, 805)) v[k] = pool[src_s[i] + off[k]];
#pragma unroll
            for (int k = 0; k < K; ++k)
                if (has[k] && SV_INB(dst_s[i] + off[k], pool_vec, 806)) pool[dst_s[i] + off[k]] = v[k];
        }
    }
    if (first) committed_out[b] = c + L + 1;
}

}  // namespace svkv

namespace sv {
// This module's first range violation (debug builds; 0 otherwise), cleared when read.
unsigned long long kv_debug_fault()
{
#ifdef SV_DEBUG
    unsigned long long w = 0, z = 0;
    if (cudaMemcpyFromSymbol(&w, g_sv_debug_fault, sizeof w) != cudaSuccess ||
        cudaMemcpyToSymbol(g_sv_debug_fault, &z, sizeof z) != cudaSuccess)
        return ~0ull;
    return w;
#else
    return 0;
#endif
}
}  // namespace sv

extern "C" int spec_verify_kv_compact(void *kv_pool, int64_t num_slots, size_t row_bytes, int planes,
                                      size_t plane_stride_bytes, const int32_t *slot_table, int max_pos,
                                      const int32_t *committed_in, int32_t *committed_out,
                                      const int32_t *accept_index, const int32_t *accept_len, int B,
                                      int N, int32_t *dev_status, void *stream)
{
    if (!kv_pool || !slot_table || !committed_in || !committed_out || !accept_index || !accept_len)
        return SPEC_VERIFY_EINVAL;
    if (committed_in == committed_out) return SPEC_VERIFY_EINVAL;
    if (B < 1 || B > 65535 || N < 1 || N > svkv::MAX_NODES || max_pos < N || num_slots < 1 || planes < 1)
        return SPEC_VERIFY_EINVAL;
    if (row_bytes == 0 || row_bytes % 16 || (uintptr_t)kv_pool % 16) return SPEC_VERIFY_EINVAL;
    if (planes > 1 && (plane_stride_bytes % 16 || plane_stride_bytes / row_bytes < (size_t)num_slots))
        return SPEC_VERIFY_EINVAL;
    const int64_t row_vec = (int64_t)(row_bytes / 16);
    const int64_t plane_vec = planes > 1 ? (int64_t)(plane_stride_bytes / 16) : 0;
    const int64_t work = row_vec * planes;
    const int64_t chunks = (work + svkv::CHUNK - 1) / svkv::CHUNK;
    if (chunks > 0x7fffffff) return SPEC_VERIFY_EINVAL;
    dim3 grid((unsigned)chunks, (unsigned)B);
    const int64_t pool_vec = (int64_t)(planes - 1) * plane_vec + num_slots * row_vec;
    svkv::kv_compact_kernel<<<grid, svkv::NT, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4 *>(kv_pool), num_slots, row_vec, plane_vec, work, pool_vec, slot_table, max_pos,
        committed_in, committed_out, accept_index, accept_len, N, dev_status);
    return cudaGetLastError() == cudaSuccess ? SPEC_VERIFY_OK : SPEC_VERIFY_ECUDA;
}
