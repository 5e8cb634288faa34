// sv_decide.cuh -- the acceptance decision of one request, taken by one warp once every row's
// statistics are known: the first-reject scan of a chain (warp ballots over 32 draft slots at a
// time), block verification's largest passing prefix, or the walk down a tree.
//
// FS is the caller's per-request state in shared memory (the finalising CTA's or a warp's); it
// provides status, tok, u, qx, node_p, row_arg, row_z, first_child, next_sib (inputs) and path,
// L, stop, mode (outputs).
#pragma once

#include "sv_device.cuh"

namespace sv {

// Chain: the first draft slot that is not accepted stops the round (warp ballots over 32 slots at
// a time).  Every lane of the calling warp gets the stop slot; it only reads F, so any number of
// warps may call it at once.
template <bool SAMPLE, bool VAR, typename FS>
__device__ __forceinline__ int chain_stop(const Params &P, const FS &F, int lane)
{
    const int k = P.k;
    for (int c0 = 0; c0 < k; c0 += 32) {
        const int i = c0 + lane;
        bool acc = false;
        if (i < k) {
            const int x = F.tok[i + 1];
            if (x >= 0) {
                if (SAMPLE && (P.q || !VAR)) {
                    acc = F.u[i] * F.qx[i + 1] < F.node_p[i + 1];
                } else if (SAMPLE) {
                    // Target-only: one candidate; thresholds of 1 give u < p(x).
                    const float px = F.node_p[i + 1];
                    acc = px > 0.f && (F.u[i] * P.thr_acc < px || px >= P.thr_single);
                } else {
                    acc = (x == F.row_arg[i]);
                }
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, i < k && !acc);
        if (m) return c0 + __ffs(m) - 1;
    }
    return k;
}

// What the round emits at a chain's stop slot j: 0 the argmax, 1 a draw from the stop row, 2 a
// residual draw left to the residual kernel (a rejected draft with draft probabilities).
template <bool SAMPLE, typename FS>
__device__ __forceinline__ int chain_mode(const Params &P, const FS &F, int j)
{
    if (!SAMPLE) return 0;
    return (j < P.k && F.tok[j + 1] >= 0 && P.q) ? 2 : 1;
}

// Decide the accepted path and the stop node (warp 0 calls it; the tree walk runs in lane 0).
// VAR: the relaxed thresholds may differ from 1.
template <bool SAMPLE, bool VAR, typename FS>
__device__ void decide_request(const Params &P, FS &F, int lane)
{
    if (F.status == 0) {
        if (SAMPLE && !P.is_tree && P.block && !P.q) {
            // Block verification with one-hot drafts (Sun et al.; "The speculative decoding zoo",
            // block branch of the rejection sampler): the prefix of L drafts has joint weight
            // w_L = prod_{i<L} p_i(x_{i+1}); candidate length L passes iff u_{L-1} < h_L, where
            // h_L = r_L / (r_L + 1 - w_L) with r_L = w_L * (the non-child share of row L) below
            // the last present draft, and h = w there.  The largest passing L is accepted.
            const int k = P.k;
            int ke = k;  // drafts present: an absent draft ends the block
            for (int c0 = 0; c0 < k; c0 += 32) {
                const unsigned m = __ballot_sync(0xffffffffu, c0 + lane < k && F.tok[c0 + lane + 1] < 0);
                if (m) {
                    ke = c0 + __ffs(m) - 1;
                    break;
                }
            }
            float wcarry = 1.f;
            int j = 0;
            for (int c0 = 0; c0 < ke; c0 += 32) {
                const int i = c0 + lane, L = i + 1;
                float w = i < ke ? F.node_p[i + 1] : 1.f;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, w, off);
                    if (lane >= off) w *= y;
                }
                w *= wcarry;  // w_L
                bool pass = false;
                if (i < ke) {
                    float h = w;
                    if (L < ke) {
                        const float r = w * F.row_z[L];
                        const float denom = r + 1.f - w;
                        h = denom > 0.f ? r / denom : 1.f;
                    }
                    pass = F.u[i] < h;
                }
                const unsigned m = __ballot_sync(0xffffffffu, pass);
                if (m) j = c0 + 32 - __clz(m);
                wcarry = __shfl_sync(0xffffffffu, w, 31);
            }
            for (int i = lane; i < j; i += 32) F.path[i] = i + 1;
            if (lane == 0) {
                F.L = j;
                F.stop = j;
                F.mode = 1;  // the token after the prefix: p with the next draft zeroed, or p
            }
        } else if (!P.is_tree) {
            const int j = chain_stop<SAMPLE, VAR>(P, F, lane);
            for (int i = lane; i < j; i += 32) F.path[i] = i + 1;
            if (lane == 0) {
                F.L = j;
                F.stop = j;
                F.mode = chain_mode<SAMPLE>(P, F, j);
            }
        } else if (lane == 0) {
            // Tree walk: one coin per depth, children in ascending node index.
            int cur = 0, depth = 0, L = 0;
            for (;;) {
                int next = -1;
                if (SAMPLE) {
                    const float coin = F.u[depth];
                    float accp = 0.f;
                    for (int ch = F.first_child[cur]; ch >= 0; ch = F.next_sib[ch]) {
                        const float pc = F.node_p[ch];
                        accp += pc;
                        if (pc > 0.f && (VAR ? (coin * P.thr_acc < accp || pc >= P.thr_single) : coin < accp)) {
                            next = ch;
                            break;
                        }
                    }
                } else {
                    const int am = F.row_arg[cur];
                    for (int ch = F.first_child[cur]; ch >= 0; ch = F.next_sib[ch]) {
                        if (F.tok[ch] == am) {
                            next = ch;
                            break;
                        }
                    }
                }
                if (next < 0) break;
                F.path[L++] = next;
                cur = next;
                ++depth;
            }
            F.L = L;
            F.stop = cur;
            F.mode = SAMPLE ? 1 : 0;
        }
    }
}

}  // namespace sv
