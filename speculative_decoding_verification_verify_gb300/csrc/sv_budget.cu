// sv_budget.cu -- the adaptive verification budget: which draft slots of a batch to verify
// ("The speculative decoding zoo", section "The finer loop: DSpark's confidence budget": every
// (request, position) slot scores the running product of its request's confidences, a global
// top-k admits the best slots with earlier positions first on ties, and the budget maximises
// expected accepted tokens per unit of step cost; "Inference Systems Frontier: new models and
// speculative decoding", section "Deciding how much to verify by load").
//
// Four kernels.  keys_kernel: the slots' survival products (fp32, the precision the decision is
// taken in) and unique 64-bit keys whose ascending order is descending survival, then position,
// then request, with out-of-range slots last.  rank_kernel: every slot counts the keys below its
// own; the grid splits both the slots and the keys they are compared with (tiles in shared
// memory read by broadcast, four slots per thread), so the whole GPU counts, and the partial
// counts add up atomically.  scatter_kernel puts every slot at its rank, so the slots end up
// sorted without a sorting network.  pick_kernel
// (one CTA): an fp64 scan of the sorted scores, the rate (B + gain[b]) / cost[b] of every budget
// (compared by cross-multiplication, divided once at the end), the first maximum, and each
// request's admitted count (its admitted slots are leading ones: the largest admitted position
// + 1).
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"
#include "sv_check.cuh"

namespace svb {

constexpr int MAX_SLOTS = SPEC_VERIFY_BUDGET_MAX_SLOTS;
constexpr int MAX_K = 64;
constexpr int NT_RANK = 128;     // threads of a ranking CTA
constexpr int RPT = 4;           // slots a ranking thread compares with each key
constexpr int SLOTS_PER_CTA = NT_RANK * RPT;
constexpr int NT_PICK = 1024;
constexpr uint64_t OUT_OF_RANGE = 1ull << 20;  // above every (position, request) field

__device__ __forceinline__ float score_of(uint64_t key) { return __uint_as_float(~(uint32_t)(key >> 32)); }

// Ascending key order: descending survival (the sign bit dropped, so -0 ranks as 0), then
// ascending position, then ascending request; out-of-range slots after every valid one.
__global__ void keys_kernel(const float *conf, const int32_t *num_drafts, int B, int K, uint64_t *keys,
                            int32_t *rank)
{
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= B) return;
    if (!SV_INB((int64_t)r * K + K - 1, (int64_t)B * K, 901)) return;
    for (int i = 0; i < K; ++i) rank[(int64_t)r * K + i] = 0;
    const int nd = num_drafts ? min(max(num_drafts[r], 0), K) : K;
    float run = 1.f;
    for (int i = 0; i < K; ++i) {
        const float c = fminf(fmaxf(conf[(int64_t)r * K + i], 0.f), 1.f);  // NaN reads as 0
        run = run * c;
        const uint64_t low = ((uint64_t)i << 14) | (uint64_t)r;
        keys[(int64_t)r * K + i] = i < nd ? ((uint64_t)(~(__float_as_uint(run) & 0x7fffffffu)) << 32) | low
                                          : (0xffffffffull << 32) | OUT_OF_RANGE | low;
    }
}

// CTA (x, y): slots [x * SLOTS_PER_CTA, + SLOTS_PER_CTA) against keys [y * span, + span).
__global__ void __launch_bounds__(NT_RANK) rank_kernel(const uint64_t *keys, int n, int span, int32_t *rank)
{
    __shared__ uint64_t tile[NT_RANK];
    const int j0 = blockIdx.x * SLOTS_PER_CTA + threadIdx.x;
    uint64_t mine[RPT];
    int below[RPT];
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
        const int j = j0 + u * NT_RANK;
        mine[u] = j < n ? keys[j] : 0ull;
        below[u] = 0;
    }
    const int k0 = blockIdx.y * span, k1 = min(k0 + span, n);
    for (int t0 = k0; t0 < k1; t0 += NT_RANK) {
        __syncthreads();
        if (t0 + (int)threadIdx.x < k1) tile[threadIdx.x] = keys[t0 + threadIdx.x];
        __syncthreads();
        const int m = min(NT_RANK, k1 - t0);
        for (int i = 0; i < m; ++i) {
            const uint64_t t = tile[i];
#pragma unroll
            for (int u = 0; u < RPT; ++u) below[u] += t < mine[u];
        }
    }
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
        const int j = j0 + u * NT_RANK;
        if (j < n && below[u]) atomicAdd(rank + j, below[u]);
    }
}

// Keys are unique, so the ranks are a permutation.
__global__ void scatter_kernel(const uint64_t *keys, const int32_t *rank, int n, uint64_t *sorted)
{
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j < n && SV_INB(rank[j], n, 902)) sorted[rank[j]] = keys[j];
}

__device__ __forceinline__ double warp_excl_scan(double x, int lane, double &total)
{
    double incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    total = __shfl_sync(0xffffffffu, incl, 31);
    return incl - x;
}

// Is rate a = na / ca above rate b = nb / cb?  Costs are positive.
__device__ __forceinline__ bool rate_above(double na, double ca, double nb, double cb) { return na * cb > nb * ca; }

__global__ void __launch_bounds__(NT_PICK) pick_kernel(const uint64_t *sorted, int n, int B, const double *cost,
                                                       int32_t *admitted, int32_t *budget_out, double *rate_out)
{
    constexpr int NW = NT_PICK / 32;
    __shared__ double wtot[NW];
    __shared__ double wnum[NW], wcost[NW];
    __shared__ int wb[NW];
    __shared__ int n_valid;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int r = tid; r < B; r += NT_PICK) admitted[r] = 0;
    // The valid slots are a prefix of the sorted order; find its length.
    if (tid == 0) n_valid = n;
    __syncthreads();
    for (int j = tid; j < n; j += NT_PICK)
        if ((sorted[j] & OUT_OF_RANGE) && (j == 0 || !(sorted[j - 1] & OUT_OF_RANGE))) n_valid = j;
    __syncthreads();
    const int nv = n_valid;
    const int per = (nv + NT_PICK - 1) / NT_PICK;
    const int j0 = min(tid * per, nv), j1 = min(j0 + per, nv);
    double own = 0.0;
    for (int j = j0; j < j1; ++j) own += (double)score_of(sorted[j]);
    double wt;
    const double wex = warp_excl_scan(own, lane, wt);
    if (lane == 0) wtot[warp] = wt;
    __syncthreads();
    double gain = wex;
    for (int w = 0; w < warp; ++w) gain += wtot[w];
    // Budgets this thread owns: b = j + 1 for its slots, and b = 0 for thread 0; first maximum.
    double bn = 0.0, bc = 1.0;
    int bb = -1;
    if (tid == 0) {
        bn = (double)B;
        bc = cost[0];
        bb = 0;
    }
    for (int j = j0; j < j1; ++j) {
        gain += (double)score_of(sorted[j]);
        const double num = (double)B + gain, c = SV_INB(j + 1, n + 1, 903) ? cost[j + 1] : 1.0;
        if (bb < 0 || rate_above(num, c, bn, bc)) {
            bn = num;
            bc = c;
            bb = j + 1;
        }
    }
    for (int round = 0; round < 2; ++round) {
        if (round == 1) {
            __syncthreads();
            if (warp != 0) break;
            bn = wnum[lane];
            bc = wcost[lane];
            bb = wb[lane];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const double on = __shfl_xor_sync(0xffffffffu, bn, o), oc = __shfl_xor_sync(0xffffffffu, bc, o);
            const int ob = __shfl_xor_sync(0xffffffffu, bb, o);
            if (ob >= 0 && (bb < 0 || rate_above(on, oc, bn, bc) || (!rate_above(bn, bc, on, oc) && ob < bb))) {
                bn = on;
                bc = oc;
                bb = ob;
            }
        }
        if (round == 0 && lane == 0) {
            wnum[warp] = bn;
            wcost[warp] = bc;
            wb[warp] = bb;
        }
    }
    if (tid == 0) {
        wb[0] = bb;
        *budget_out = bb;
        if (rate_out) *rate_out = bn / bc;
    }
    __syncthreads();
    const int budget = wb[0];
    for (int j = tid; j < budget; j += NT_PICK) {
        const uint32_t lo = (uint32_t)sorted[j];
        if (SV_INB(lo & 0x3fffu, B, 904)) atomicMax(admitted + (lo & 0x3fffu), (int)((lo >> 14) & 0x3fu) + 1);
    }
}

}  // namespace svb

namespace sv {
// This module's first range violation (debug builds; 0 otherwise), cleared when read.
unsigned long long budget_debug_fault()
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

extern "C" size_t spec_verify_plan_budget_workspace_bytes(int B, int K)
{
    if (B < 1 || K < 1 || K > svb::MAX_K || (int64_t)B * K > svb::MAX_SLOTS) return 0;
    return (2 * sizeof(uint64_t) + sizeof(int32_t)) * (size_t)B * (size_t)K;
}

extern "C" int spec_verify_plan_budget(const float *conf, const int32_t *num_drafts, int B, int K,
                                       const double *cost, int32_t *admitted, int32_t *budget,
                                       double *best_rate, void *workspace, size_t ws_bytes, void *stream)
{
    if (!conf || !cost || !admitted || !budget || !workspace) return SPEC_VERIFY_EINVAL;
    if (B < 1 || K < 1 || K > svb::MAX_K || (int64_t)B * K > svb::MAX_SLOTS) return SPEC_VERIFY_EINVAL;
    if ((uintptr_t)conf % 4 || (uintptr_t)cost % 8 || (uintptr_t)admitted % 4 || (uintptr_t)budget % 4 ||
        (uintptr_t)num_drafts % 4 || (uintptr_t)best_rate % 8)
        return SPEC_VERIFY_EINVAL;
    const int n = B * K;
    if ((uintptr_t)workspace % 8 || ws_bytes < spec_verify_plan_budget_workspace_bytes(B, K))
        return SPEC_VERIFY_EWORKSPACE;
    uint64_t *keys = static_cast<uint64_t *>(workspace);
    uint64_t *sorted = keys + n;
    int32_t *rank = reinterpret_cast<int32_t *>(sorted + n);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    svb::keys_kernel<<<(B + 255) / 256, 256, 0, s>>>(conf, num_drafts, B, K, keys, rank);
    // Split the keys each slot is compared with until about 1024 CTAs count at once.
    const int gx = (n + svb::SLOTS_PER_CTA - 1) / svb::SLOTS_PER_CTA;
    int gy = (1024 + gx - 1) / gx;
    const int max_gy = (n + svb::NT_RANK - 1) / svb::NT_RANK;
    if (gy > max_gy) gy = max_gy;
    const int span = ((n + gy - 1) / gy + svb::NT_RANK - 1) / svb::NT_RANK * svb::NT_RANK;
    gy = (n + span - 1) / span;
    svb::rank_kernel<<<dim3(gx, gy), svb::NT_RANK, 0, s>>>(keys, n, span, rank);
    svb::scatter_kernel<<<(n + 255) / 256, 256, 0, s>>>(keys, rank, n, sorted);
    svb::pick_kernel<<<1, svb::NT_PICK, 0, s>>>(sorted, n, B, cost, admitted, budget, best_rate);
    return cudaGetLastError() == cudaSuccess ? SPEC_VERIFY_OK : SPEC_VERIFY_ECUDA;
}
