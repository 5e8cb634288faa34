// spec_verify.cu -- the batched speculative-decoding verifier for GB300 (sm_103a), behind the
// C ABI declared in include/spec_verify.h.
//
// Hot path ("投机解码" [Speculative decoding], rustineverything, sections 目标模型怎么一次验证 and
// 接受规则为什么不改变分布; "The speculative decoding zoo", mlinterviewnotes 06-06, DFlash and
// verification-method sections):
//
//   sv_stream_kernel   -- one pass over all B * rows * V logits.  The flat range is split evenly
//                         over G persistent CTAs.  Each warp keeps a running (max, sum of
//                         2^(l*cs - max*cs)) over its contiguous segment, skipping the tokens
//                         that are drafts of the row (their logits are captured instead), or a
//                         running argmax (greedy), and writes one record per piece.
//   sv_finalize_kernel -- one CTA per request, launched as a programmatic dependent of the
//                         streaming kernel: it stages the request's inputs, waits for the records,
//                         merges them per row, decides acceptance (warp-ballot first-reject scan
//                         for chains, a walk for trees), and draws the stop token by locating the
//                         record whose running mass crosses v * Z and rescanning only that segment.
//   sv_residual_kernel -- standard rejection only: at the rejected row j, the draw comes from
//                         max(0, p - q); its normaliser needs the row's full softmax sum, so the
//                         logits and q of row j are read once more, split over CTAs; the last CTA
//                         of a request (atomic arrival counter, nothing waits) draws.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "spec_verify.h"
#include "sv_device.cuh"
#include "sv_draw.cuh"
#include "sv_stream.cuh"
#include "sv_rescan.cuh"

namespace sv {

#ifndef SV_MINB
#define SV_MINB 3
#endif
constexpr int NT_FIN = 256;    // threads of a finalising CTA
#ifndef SV_CTAS_PER_SM
#define SV_CTAS_PER_SM 0  // streaming CTAs per SM (0: as many as fit)
#endif

struct StreamSmem {
    int ex_col[MAX_RPR];   // sorted columns of the current row's child tokens
    int ex_node[MAX_RPR];  // the child node of each
    int ex_cnt;
    int last;
};

struct FinSmem {
    int par[MAX_RPR], tok[MAX_RPR];
    int first_child[MAX_RPR], next_sib[MAX_RPR];
    float row_mc[MAX_RPR], row_S[MAX_RPR], row_tot[MAX_RPR];
    float node_e[MAX_RPR], node_p[MAX_RPR], qx[MAX_RPR], capl[MAX_RPR];
    float u[MAX_RPR], v[MAX_RPR];
    float row_best[MAX_RPR];
    int row_arg[MAX_RPR];
    int acc[MAX_RPR];
    int path[MAX_RPR];
    int status;
    int stop;     // node at which the round stops
    int L;        // accepted drafts
    int mode;     // 0 emit argmax, 1 draw from the stop row (children zeroed), 2 residual pending
    int take_last;
    int rec;
    float cum_before;
    float thresh;
    int last_tok;
    int ex_col[MAX_RPR];
    int ex_cnt;
    DrawSmem D;
    RescanSmem RS;
};

struct Smem {
    StreamSmem st;
    FinSmem fin;
};

// ---------------------------------------------------------------------------------------------
// Children of node n with a usable token, sorted by token column (warp 0 builds it).
// ---------------------------------------------------------------------------------------------
__device__ void build_children(const Params &P, int b, int n, int *ex_col, int *ex_node,
                               int *ex_cnt, int lane)
{
    int cnt = 0;
    for (int base = n + 1; base < P.rpr; base += 32) {
        const int ch = base + lane;
        bool ok = false;
        int tok = -1;
        if (ch < P.rpr) {
            const int pa = node_parent(P, b, ch);
            tok = node_token(P, b, ch);
            ok = (pa == n) && tok >= 0 && (int64_t)tok < P.V;
        }
        const unsigned m = __ballot_sync(0xffffffffu, ok);
        if (ok) {
            const int pos = cnt + __popc(m & ((1u << lane) - 1u));
            ex_col[pos] = tok;
            ex_node[pos] = ch;
        }
        cnt += __popc(m);
    }
    __syncwarp();
    if (lane == 0) {
        for (int i = 1; i < cnt; ++i) {  // insertion sort by column (few entries)
            const int c = ex_col[i], nd = ex_node[i];
            int j = i - 1;
            while (j >= 0 && ex_col[j] > c) {
                ex_col[j + 1] = ex_col[j];
                ex_node[j + 1] = ex_node[j];
                --j;
            }
            ex_col[j + 1] = c;
            ex_node[j + 1] = nd;
        }
        *ex_cnt = cnt;
    }
    __syncwarp();
}

// The same child list, built by the finalising CTA from the structure it staged in shared memory.
__device__ void children_from_smem(FinSmem &F, int n, int rpr, int64_t V, int *ex_node, int lane)
{
    int cnt = 0;
    for (int base = n + 1; base < rpr; base += 32) {
        const int ch = base + lane;
        const bool ok = ch < rpr && F.par[ch] == n && F.tok[ch] >= 0 && (int64_t)F.tok[ch] < V;
        const unsigned m = __ballot_sync(0xffffffffu, ok);
        if (ok) {
            const int pos = cnt + __popc(m & ((1u << lane) - 1u));
            F.ex_col[pos] = F.tok[ch];
            ex_node[pos] = ch;
        }
        cnt += __popc(m);
    }
    __syncwarp();
    if (lane == 0) {
        for (int i = 1; i < cnt; ++i) {
            const int c = F.ex_col[i], nd = ex_node[i];
            int j = i - 1;
            while (j >= 0 && F.ex_col[j] > c) {
                F.ex_col[j + 1] = F.ex_col[j];
                ex_node[j + 1] = ex_node[j];
                --j;
            }
            F.ex_col[j + 1] = c;
            ex_node[j + 1] = nd;
        }
        F.ex_cnt = cnt;
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------------------------
// One warp streams its segment [c0, c1) of a row: the unaligned head and tail element by element,
// the 16-byte aligned body with vector loads.  Each lane visits its columns in ascending order.
// ---------------------------------------------------------------------------------------------
template <typename T, bool SAMPLE>
__device__ __forceinline__ void stream_segment(const T *row, const Seg &sg, int lane, float cs,
                                               ExCursor &ex, SampleAcc &sa, GreedyAcc &ga)
{
    for (int c = (int)sg.c0 + lane; c < (int)sg.b0; c += 32) {
        const float x = Elt<T>::load(row, c);
        if (SAMPLE) sample_scalar(sa, x, c, cs, ex);
        else greedy_scalar(ga, x, c);
    }
    stream_body<T, SAMPLE>(row, (int)sg.b0, (int)sg.b1, lane, cs, ex, sa, ga);
    for (int c = (int)sg.b1 + lane; c < (int)sg.c1; c += 32) {
        const float x = Elt<T>::load(row, c);
        if (SAMPLE) sample_scalar(sa, x, c, cs, ex);
        else greedy_scalar(ga, x, c);
    }
}

// ---------------------------------------------------------------------------------------------
// Draw sources for the block rescan.
// ---------------------------------------------------------------------------------------------
// Body of a segment: one 16-byte vector per group; weight 2^(l*cs - mc), children zeroed.
template <typename T>
struct VecSrc {
    static constexpr int GS = Elt<T>::VEC;
    using Raw = uint4;
    const uint4 *vp;
    int64_t col0;  // column of group 0
    float cs, mc;
    const int *ex;
    int ex_cnt;
    __device__ Raw prefetch(int64_t gi) const { return ldg_stream(vp + gi); }
    __device__ int weights(const Raw &r, int64_t gi, float (&w)[GS]) const
    {
        float x[GS];
        Elt<T>::unpack(r, x);
        const int c = (int)(col0 + gi * GS);
#pragma unroll
        for (int j = 0; j < GS; ++j) w[j] = ex2(fmaf(x[j], cs, -mc));
        for (int e = 0; e < ex_cnt; ++e) {
            const int d = ex[e] - c;
#pragma unroll
            for (int j = 0; j < GS; ++j)
                if (d == j) w[j] = 0.f;
        }
        return c;
    }
};

// Unaligned head or tail: one element per group.
template <typename T>
struct ScalarSrc {
    static constexpr int GS = 1;
    using Raw = float;
    const void *row;
    int64_t col0;
    float cs, mc;
    const int *ex;
    int ex_cnt;
    __device__ Raw prefetch(int64_t gi) const { return Elt<T>::load(row, col0 + gi); }
    __device__ int weights(const Raw &x, int64_t gi, float (&w)[1]) const
    {
        const int c = (int)(col0 + gi);
        w[0] = ex2(fmaf(x, cs, -mc));
        for (int e = 0; e < ex_cnt; ++e)
            if (ex[e] == c) w[0] = 0.f;
        return c;
    }
};

__device__ __forceinline__ void draw_init(DrawSmem &D, float cum)
{
    if (threadIdx.x == 0) {
        D.cum = cum;
        D.found = -1;
        D.lastpos = -1;
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------------------------
// Finalisation of request b by the last CTA to finish it.
// ---------------------------------------------------------------------------------------------
extern __shared__ __align__(16) unsigned char sv_dyn_smem[];

template <typename T, bool SAMPLE, int NTF>
__device__ void finalize_request(const Params &P, int b, Smem &sm)
{
    FinSmem &F = sm.fin;
    constexpr int NWF = NTF / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rpr = P.rpr;
    const int64_t V = P.V;
    const int64_t rbase = (int64_t)b * rpr;

    // Prologue on inputs only (may overlap the streaming kernel): structure, q(x), uniforms.
    for (int n = tid; n < rpr; n += NTF) {
        F.par[n] = n == 0 ? (P.is_tree ? __ldg(P.parents + rbase) : -1) : node_parent(P, b, n);
        F.tok[n] = n == 0 ? -1 : node_token(P, b, n);
        float qv = 1.f;
        if (SAMPLE && P.q && n >= 1 && n <= P.k) {
            const int x = F.tok[n];
            if (x >= 0 && (int64_t)x < V) qv = __ldg(P.q + ((int64_t)b * P.k + (n - 1)) * V + x);
        }
        F.qx[n] = qv;
        if (SAMPLE) {
            const float2 uv = uniforms(P, (uint32_t)n, (uint32_t)b);
            F.u[n] = uv.x;
            F.v[n] = uv.y;
        }
    }
    if (tid == 0) F.status = 0;
    __syncthreads();

    // Window of record indices covering all rows of the request (contiguous, possibly with unused
    // slots); small enough windows are kept in shared memory for the draw's locate step.
    const int64_t win0 = (rbase * V / P.E + rbase) * NW;
    const int64_t win1 = (((rbase + rpr) * V - 1) / P.E + rbase + rpr - 1) * NW + NW;
    float2 *recs_s = reinterpret_cast<float2 *>(sv_dyn_smem);
    const bool keep = SAMPLE && (win1 - win0) * (int64_t)sizeof(float2) <= (int64_t)RESCAN_SMEM_BYTES;

    // From here on the streaming kernel's records and captures are read.
    pdl_wait();
    // Captured logits of each node's token in its parent's row, and the per-row merge of the
    // warp records (one warp per row); all these loads are in flight together.
    for (int n = tid; n < rpr; n += NTF) {
        float l = NEG_INF;
        if (SAMPLE && n >= 1) {
            const int pa = F.par[n], tk = F.tok[n];
            if (pa >= 0 && pa < n && tk >= 0 && (int64_t)tk < V) l = __ldcg(P.caps + rbase + n);
        }
        F.capl[n] = l;
    }
    for (int i = warp; i < rpr; i += NWF) {
        const int64_t r = rbase + i;
        const int64_t rowf = r * V;
        const int64_t g_lo = rowf / P.E, g_hi = (rowf + V - 1) / P.E;
        const int64_t base = (g_lo + r) * NW;
        const int L = (int)((g_hi - g_lo + 1) * NW);
        if (SAMPLE) {
            float mc = REF_NONE, s = 0.f;
            for (int t = lane; t < L; t += 32) {
                const float2 rec = __ldcg(P.recs + base + t);
                if (keep) recs_s[base + t - win0] = rec;
                rec_merge(mc, s, rec.x, rec.y);
            }
            warp_rec_merge(mc, s);
            if (lane == 0) {
                F.row_mc[i] = mc;
                F.row_S[i] = s;
            }
        } else {
            float best = NEG_INF;
            int idx = INT_MAX;
            for (int t = lane; t < L; t += 32) {
                const float2 rec = __ldcg(P.recs + base + t);
                arg_merge(best, idx, rec.x, __float_as_int(rec.y));
            }
            warp_arg_merge(best, idx);
            if (lane == 0) {
                F.row_best[i] = best;
                F.row_arg[i] = idx;
            }
        }
    }
    __syncthreads();

    // Validation; the largest fault code of the request wins.
    {
        int st = 0;
        for (int n = tid; n < rpr; n += NTF) {
            if (n >= 1) {
                const int tk = F.tok[n];
                if (tk < -1 || (int64_t)tk >= V) st = max(st, SPEC_VERIFY_DEV_BAD_TOKEN);
                if (P.is_tree && (F.par[n] < 0 || F.par[n] >= n)) st = max(st, SPEC_VERIFY_DEV_BAD_TREE);
                if (P.is_tree && SAMPLE && tk >= 0) {
                    for (int m = n + 1; m < rpr; ++m)
                        if (F.par[m] == F.par[n] && F.tok[m] == tk) st = max(st, SPEC_VERIFY_DEV_DUP_SIBLING);
                }
            } else if (P.is_tree && F.par[0] != -1) {
                st = max(st, SPEC_VERIFY_DEV_BAD_TREE);
            }
            bool bad;
            if (SAMPLE) {
                bad = !(fabsf(F.row_mc[n]) < POS_INF) || !(F.row_S[n] >= 0.f) || !(F.row_S[n] < POS_INF);
            } else {
                const float bv = F.row_best[n];
                bad = !(fabsf(bv) < POS_INF);
            }
            if (bad) st = max(st, SPEC_VERIFY_DEV_BAD_ROW);
        }
        if (st) atomicMax(&F.status, st);
    }
    // Children lists (ascending node index) and, when sampling, each child's probability.
    for (int n = tid; n < rpr; n += NTF) {
        int fc = -1, ns = -1;
        for (int m = n + 1; m < rpr; ++m) {
            if (fc < 0 && F.par[m] == n && F.tok[m] >= 0) fc = m;
        }
        if (n >= 1) {
            for (int m = n + 1; m < rpr; ++m) {
                if (F.par[m] == F.par[n] && F.tok[m] >= 0) {
                    ns = m;
                    break;
                }
            }
        }
        F.first_child[n] = fc;
        F.next_sib[n] = ns;
        if (SAMPLE && n >= 1) {
            const int pa = F.par[n], tk = F.tok[n];
            float e = 0.f;
            if (pa >= 0 && pa < n && tk >= 0 && (int64_t)tk < V) e = ex2(fmaf(F.capl[n], P.cs, -F.row_mc[pa]));
            F.node_e[n] = e;
        }
    }
    __syncthreads();
    if (SAMPLE) {
        for (int n = tid; n < rpr; n += NTF) {
            float extra = 0.f;
            for (int m = n + 1; m < rpr; ++m)
                if (F.par[m] == n && F.tok[m] >= 0 && (int64_t)F.tok[m] < V) extra += F.node_e[m];
            F.row_tot[n] = F.row_S[n] + extra;
        }
        __syncthreads();
        for (int n = 1 + tid; n < rpr; n += NTF) {
            const int pa = F.par[n];
            F.node_p[n] = (pa >= 0 && pa < n) ? F.node_e[n] / F.row_tot[pa] : 0.f;
        }
        if (tid < rpr) {
            const float tot = F.row_tot[tid];
            if (!(tot > 0.f) || !(tot < POS_INF)) atomicMax(&F.status, SPEC_VERIFY_DEV_BAD_ROW);
        }
        __syncthreads();
    }

    // Decide the accepted path and the stop node.
    const bool faulted = F.status != 0;
    if (!faulted) {
        if (!P.is_tree) {
            // Chain: acc[i] for draft slot i; the first non-accepted slot stops the round.
            const int k = P.k;
            if (tid < 64) {
                bool acc = false;
                if (tid < k) {
                    const int x = F.tok[tid + 1];
                    if (x >= 0) {
                        if (SAMPLE) acc = F.u[tid] * F.qx[tid + 1] < F.node_p[tid + 1];
                        else acc = (x == F.row_arg[tid]);
                    }
                }
                const unsigned m = __ballot_sync(0xffffffffu, !acc);
                if (lane == 0) F.acc[warp] = (int)m;  // warps 0 and 1 cover slots 0..63
            }
            __syncthreads();
            if (tid == 0) {
                const unsigned m0 = (unsigned)F.acc[0];
                const unsigned m1 = (unsigned)F.acc[1];
                int j = m0 ? (__ffs(m0) - 1) : (32 + __ffs(m1) - 1);
                if (j > k) j = k;
                F.L = j;
                F.stop = j;
                for (int i = 0; i < j; ++i) F.path[i] = i + 1;
                if (!SAMPLE) F.mode = 0;
                else if (j < k && F.tok[j + 1] >= 0 && P.q) F.mode = 2;
                else F.mode = 1;
            }
        } else if (tid == 0) {
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
                        if (pc > 0.f && coin < accp) {
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
    __syncthreads();

    // Draw the stop token from row `stop`, children zeroed (they were tried), unless the
    // draw is the standard-rejection residual, which the residual kernel does.
    int drawn = -1;
    if (!faulted && F.mode == 1) {
        const int n = F.stop;
        const int64_t r = rbase + n;
        const float mc_r = F.row_mc[n];
        const float vdraw = F.v[P.is_tree ? F.L : n];
        if (warp == 0) children_from_smem(F, n, rpr, V, sm.st.ex_node, lane);
        __syncthreads();
        if (F.row_S[n] > 0.f) {
            const float t = vdraw * F.row_S[n];
            // Locate the record holding the crossing (warp 0).
            const int64_t rowf = r * V;
            const int64_t g_lo = rowf / P.E, g_hi = (rowf + V - 1) / P.E;
            const int64_t base = (g_lo + r) * NW;
            const int L = (int)((g_hi - g_lo + 1) * NW);
            if (warp == 0) {
                float cum = 0.f, before = 0.f, lp_before = 0.f;
                int found = -1, lastpos = -1;
                for (int c = 0; c < L; c += 32) {
                    const int ti = c + lane;
                    float m = 0.f;
                    if (ti < L) {
                        const float2 rec = keep ? recs_s[base + ti - win0] : __ldcg(P.recs + base + ti);
                        m = (rec.y == 0.f) ? 0.f : rec.y * ex2(rec.x - mc_r);
                    }
                    const float incl = warp_incl_scan(m, lane);
                    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                    if (lane == 0) excl = 0.f;
                    const unsigned hit = __ballot_sync(0xffffffffu, cum + incl > t);
                    const unsigned pos = __ballot_sync(0xffffffffu, m > 0.f);
                    if (pos) {
                        const int lp = 31 - __clz(pos);
                        lastpos = c + lp;
                        lp_before = cum + __shfl_sync(0xffffffffu, excl, lp);
                    }
                    if (hit) {
                        const int fl = __ffs(hit) - 1;
                        found = c + fl;
                        before = cum + __shfl_sync(0xffffffffu, excl, fl);
                        break;
                    }
                    cum += __shfl_sync(0xffffffffu, incl, 31);
                }
                if (lane == 0) {
                    if (found >= 0) {
                        F.rec = found;
                        F.cum_before = before;
                        F.take_last = 0;
                    } else {
                        F.rec = lastpos;
                        F.cum_before = lp_before;
                        F.take_last = 1;
                    }
                }
            }
            __syncthreads();
            const int rec = F.rec;
            if (rec >= 0) {
                const int64_t g = g_lo + rec / NW;
                const int w = rec % NW;
                const Seg sg = seg_of<Elt<T>::VEC>(P, g, r, w);
                const float tt = F.take_last ? POS_INF : t;
                const T *row = reinterpret_cast<const T *>(P.logits) + r * V;
                drawn = rescan_segment<T, NTF>(row, sg, P.cs, mc_r, tt, F.cum_before, F.ex_col, F.ex_cnt,
                                               sv_dyn_smem, F.RS);
            }
        } else {
            // Every non-child token underflowed: draw among the children, by p, in column order.
            if (tid == 0) {
                float tot = 0.f;
                for (int e = 0; e < F.ex_cnt; ++e) tot += F.node_e[sm.st.ex_node[e]];
                const float t = vdraw * tot;
                float c = 0.f;
                for (int e = 0; e < F.ex_cnt && drawn < 0; ++e) {
                    const float w = F.node_e[sm.st.ex_node[e]];
                    if (w > 0.f) {
                        c += w;
                        if (c > t) drawn = F.ex_col[e];
                    }
                }
                if (drawn < 0 && F.ex_cnt > 0) drawn = F.ex_col[F.ex_cnt - 1];
            }
        }
    }
    if (tid == 0) {
        int last = -1;
        if (!faulted) {
            if (F.mode == 0) last = F.row_arg[F.stop];
            else if (F.mode == 1) last = drawn >= 0 ? drawn : 0;  // < 0 only through rounding
        }
        F.last_tok = last;
    }
    __syncthreads();

    // Outputs.
    const int out_w = P.is_tree ? rpr : P.k + 1;
    int32_t *ot = P.out_tokens + (int64_t)b * out_w;
    if (faulted) {
        for (int i = tid; i < out_w; i += NTF) {
            ot[i] = -1;
            if (P.is_tree) P.accept_index[(int64_t)b * rpr + i] = -1;
        }
        if (tid == 0) {
            P.accept_len[b] = -1;
            raise_status(P.dev_status, F.status);
        }
        if (SAMPLE && P.out_probs && !P.is_tree)
            for (int i = tid; i < (P.k + 1) * 3; i += NTF) P.out_probs[(int64_t)b * (P.k + 1) * 3 + i] = 0.f;
        if (SAMPLE && P.q && !P.is_tree && tid == 0) P.pend[b] = make_int4(-1, 0, 0, 0);
    } else {
        const int L = F.L;
        for (int i = tid; i < out_w; i += NTF) {
            int v = -1;
            if (i < L) v = F.tok[F.path[i]];
            else if (i == L) v = F.last_tok;
            ot[i] = v;
            if (P.is_tree) P.accept_index[(int64_t)b * rpr + i] = (i == 0) ? 0 : (i <= L ? F.path[i - 1] : -1);
        }
        if (tid == 0) {
            P.accept_len[b] = L;
            if (SAMPLE && P.q && !P.is_tree) {
                if (F.mode == 2) {
                    const int n = F.stop;
                    P.pend[b] = make_int4(n, __float_as_int(F.row_mc[n]), __float_as_int(F.row_tot[n]), 1);
                } else {
                    P.pend[b] = make_int4(-1, 0, 0, 0);
                }
            }
        }
        if (SAMPLE && P.out_probs && !P.is_tree) {
            float *op = P.out_probs + (int64_t)b * (P.k + 1) * 3;
            for (int i = tid; i <= P.k; i += NTF) {
                float p0 = 0.f, q0 = 0.f, z = 0.f;
                if (i < P.k && F.tok[i + 1] >= 0) {
                    p0 = F.node_p[i + 1];
                    q0 = F.qx[i + 1];
                }
                if (i == F.stop && F.mode == 1) z = F.row_S[i] / F.row_tot[i];
                op[3 * i + 0] = p0;
                op[3 * i + 1] = q0;
                op[3 * i + 2] = z;
            }
        }
    }
}

// ---------------------------------------------------------------------------------------------
// The streaming kernel: every CTA folds its share of the flat logits range into per-warp records.
// ---------------------------------------------------------------------------------------------
template <typename T, bool SAMPLE>
__global__ void __launch_bounds__(NT, SV_MINB) sv_stream_kernel(const Params P)
{
    __shared__ StreamSmem st;
    constexpr int VEC = Elt<T>::VEC;
    const int g = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t V = P.V;
    const int64_t F0 = (int64_t)g * P.E;
    const int64_t F1 = min(F0 + P.E, P.total);
    pdl_launch_dependents();
    if (F0 >= F1) return;
    const int64_t r_end = (F1 - 1) / V;
    for (int64_t r = F0 / V; r <= r_end; ++r) {
        const int b = (int)(r / P.rpr);
        const int n = (int)(r - (int64_t)b * P.rpr);
        if (SAMPLE) {
            __syncthreads();
            if (warp == 0) build_children(P, b, n, st.ex_col, st.ex_node, &st.ex_cnt, lane);
            __syncthreads();
        }
        const Seg sg = seg_of<VEC>(P, g, r, warp);
        const T *row = reinterpret_cast<const T *>(P.logits) + r * V;
        SampleAcc sa;
        GreedyAcc ga;
        ExCursor ex;
        ex.init(st.ex_col, st.ex_node, SAMPLE ? st.ex_cnt : 0, P.caps + (int64_t)b * P.rpr);
        stream_segment<T, SAMPLE>(row, sg, lane, P.cs, ex, sa, ga);
        float2 rec;
        if (SAMPLE) {
            float mc = sa.mc, sum = sa.total();
            warp_rec_merge(mc, sum);
            rec = make_float2(mc, sum);
        } else {
            warp_arg_merge(ga.best, ga.idx);
            rec = make_float2(ga.best, __int_as_float(ga.idx));
        }
        if (lane == 0) P.recs[(g + r) * NW + warp] = rec;
    }
    (void)tid;
}

// ---------------------------------------------------------------------------------------------
// The finalising kernel: one CTA per request merges its records, decides and draws.
// ---------------------------------------------------------------------------------------------
template <typename T, bool SAMPLE>
__global__ void __launch_bounds__(NT_FIN) sv_finalize_kernel(const Params P)
{
    __shared__ Smem sm;
    finalize_request<T, SAMPLE, NT_FIN>(P, (int)blockIdx.x, sm);
}

// ---------------------------------------------------------------------------------------------
// Residual kernel (standard rejection): draw from max(0, p - q) at the rejected row.
// Grid (C2, B).  Each warp sums the residual r = max(0, p - q) and p over its part of the
// chunk; the last CTA of a request locates the crossing and rescans that part.
// ---------------------------------------------------------------------------------------------
template <typename T>
struct ResidSrc {
    static constexpr int GS = 8;
    struct Raw {
        float l[8];
        float q[8];
    };
    const void *row;
    const float *qrow;
    int64_t col0, col1;  // part [col0, col1)
    float cs, mc, inv;
    int use_p;           // draw from p instead (residual mass underflowed)
    __device__ Raw prefetch(int64_t gi) const
    {
        Raw r;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t c = col0 + gi * 8 + j;
            const bool in = c < col1;
            r.l[j] = in ? Elt<T>::load(row, c) : NEG_INF;
            r.q[j] = in ? __ldg(qrow + c) : 0.f;
        }
        return r;
    }
    __device__ int weights(const Raw &r, int64_t gi, float (&w)[8]) const
    {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float p = ex2(fmaf(r.l[j], cs, -mc)) * inv;
            w[j] = use_p ? p : fmaxf(0.f, p - r.q[j]);
        }
        return (int)(col0 + gi * 8);
    }
};

template <typename T>
__global__ void __launch_bounds__(NT) sv_residual_kernel(const Params P)
{
    __shared__ FinSmem F;
    __shared__ int is_last;
    const int c = (int)(blockIdx.x % (unsigned)P.C2), b = (int)(blockIdx.x / (unsigned)P.C2);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int4 pd = P.pend[b];
    if (pd.w != 1) return;
    const int j = pd.x;
    const float mc = __int_as_float(pd.y), tot = __int_as_float(pd.z);
    const float inv = 1.f / tot;
    const int64_t V = P.V;
    const int64_t r = (int64_t)b * P.rpr + j;
    const void *row = reinterpret_cast<const T *>(P.logits) + r * V;
    const float *qrow = P.q + ((int64_t)b * P.k + j) * V;
    const int64_t cc0 = (int64_t)c * P.Ec2, cc1 = min(cc0 + P.Ec2, V);
    const int64_t span = (cc1 - cc0 + NW - 1) / NW;
    const int64_t w0 = min(cc0 + warp * span, cc1), w1 = min(w0 + span, cc1);
    float zr = 0.f, zp = 0.f;
    for (int64_t base = w0; base < w1; base += 32 * 8) {
        float l[8], q[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int64_t col = base + lane + 32 * u;
            const bool in = col < w1;
            l[u] = in ? Elt<T>::load(row, col) : NEG_INF;
            q[u] = in ? __ldg(qrow + col) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float p = ex2(fmaf(l[u], P.cs, -mc)) * inv;
            zp += p;
            zr += fmaxf(0.f, p - q[u]);
        }
    }
    zr = warp_sum(zr);
    zp = warp_sum(zp);
    if (lane == 0) P.recs2[((int64_t)b * P.C2 + c) * NW + warp] = make_float2(zr, zp);
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned old = atomicAdd(P.cnt2 + b, 1u);
        is_last = (old == (unsigned)P.C2 - 1u);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    // Last CTA: total residual mass, then the crossing record (warp 0), then the rescan.
    const float2 *rb = P.recs2 + (int64_t)b * P.C2 * NW;
    const int L = P.C2 * NW;
    if (warp == 0) {
        float zr_t = 0.f, zp_t = 0.f;
        for (int t = lane; t < L; t += 32) {
            const float2 x = __ldcg(rb + t);
            zr_t += x.x;
            zp_t += x.y;
        }
        zr_t = warp_sum(zr_t);
        zp_t = warp_sum(zp_t);
        const int use_p = !(zr_t > 0.f);
        const float Z = use_p ? zp_t : zr_t;
        const float t = uniforms(P, (uint32_t)j, (uint32_t)b).y * Z;
        float cum = 0.f, before = 0.f, lp_before = 0.f;
        int found = -1, lastpos = -1;
        for (int c0 = 0; c0 < L; c0 += 32) {
            const int ti = c0 + lane;
            float m = 0.f;
            if (ti < L) {
                const float2 x = __ldcg(rb + ti);
                m = use_p ? x.y : x.x;
            }
            const float incl = warp_incl_scan(m, lane);
            float excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (lane == 0) excl = 0.f;
            const unsigned hit = __ballot_sync(0xffffffffu, cum + incl > t);
            const unsigned pos = __ballot_sync(0xffffffffu, m > 0.f);
            if (pos) {
                const int lp = 31 - __clz(pos);
                lastpos = c0 + lp;
                lp_before = cum + __shfl_sync(0xffffffffu, excl, lp);
            }
            if (hit) {
                const int fl = __ffs(hit) - 1;
                found = c0 + fl;
                before = cum + __shfl_sync(0xffffffffu, excl, fl);
                break;
            }
            cum += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            F.rec = found >= 0 ? found : lastpos;
            F.cum_before = found >= 0 ? before : lp_before;
            F.take_last = found < 0;
            F.thresh = t;
            F.mode = use_p;
            F.row_tot[0] = use_p ? 1.f : zr_t;
        }
    }
    __syncthreads();
    int drawn = -1;
    if (F.rec >= 0) {
        const int rc = F.rec / NW, rw = F.rec % NW;
        const int64_t a0 = (int64_t)rc * P.Ec2, a1 = min(a0 + P.Ec2, V);
        const int64_t sp = (a1 - a0 + NW - 1) / NW;
        const int64_t s0 = min(a0 + rw * sp, a1), s1 = min(s0 + sp, a1);
        ResidSrc<T> src{row, qrow, s0, s1, P.cs, mc, inv, F.mode};
        draw_init(F.D, F.cum_before);
        draw_span<2>(src, (s1 - s0 + 7) / 8, F.take_last ? POS_INF : F.thresh, F.D);
        drawn = F.D.found >= 0 ? F.D.found : F.D.lastpos;
    }
    if (tid == 0) {
        P.out_tokens[(int64_t)b * (P.k + 1) + j] = drawn >= 0 ? drawn : 0;
        if (P.out_probs) P.out_probs[((int64_t)b * (P.k + 1) + j) * 3 + 2] = F.row_tot[0];
        P.cnt2[b] = 0u;
    }
}

__global__ void sv_philox_kernel(uint32_t k0, uint32_t k1, uint32_t o0, uint32_t o1, int n_slot,
                                  int n_req, uint32_t *out)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)n_slot * n_req) return;
    const int slot = (int)(i / n_req), req = (int)(i % n_req);
    const uint4 w = philox4x32_10((uint32_t)slot, (uint32_t)req, o0, o1, k0, k1);
    reinterpret_cast<uint4 *>(out)[i] = w;
}

// ---------------------------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int residual_chunks(int B, int64_t V)
{
    const int64_t want = (1024 + B - 1) / B;
    const int64_t cap = (V + 1023) / 1024;
    int64_t c = want < cap ? want : cap;
    if (c < 1) c = 1;
    if (c > C2_MAX) c = C2_MAX;
    return (int)c;
}

struct Layout {
    size_t cnt1, cnt2, recs, caps, pend, recs2, total;
};

static Layout layout(int B, int rpr, int64_t V)
{
    // The arrival counters sit in a fixed region at the start of every layout, so a workspace
    // shared by calls of different shapes never finds another call's records where its counters
    // are: every call leaves that region zero, whatever the shape of the next call.
    const int64_t R = (int64_t)B * rpr;
    const int C2 = residual_chunks(B, V);
    Layout L;
    size_t off = 0;
    L.cnt1 = off;
    off += sizeof(unsigned) * (size_t)B_MAX;
    L.cnt2 = off;
    off += sizeof(unsigned) * (size_t)B_MAX;
    L.recs = off;
    off += align256(sizeof(float2) * (size_t)(G_MAX + R) * NW);
    L.caps = off;
    off += align256(sizeof(float) * (size_t)R);
    L.pend = off;
    off += align256(sizeof(int4) * (size_t)B);
    L.recs2 = off;
    off += align256(sizeof(float2) * (size_t)B * C2 * NW);
    L.total = off;
    return L;
}

struct DevInfo {
    int sms = 0;
    int occ[2][2] = {{0, 0}, {0, 0}};  // [dtype][sample]
};

static std::mutex g_dev_mu;
static DevInfo g_dev[64];

static const DevInfo *device_info()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo &d = g_dev[dev];
    if (d.sms == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
        int o = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sv_stream_kernel<__nv_bfloat16, false>, NT, 0);
        d.occ[0][0] = o > 0 ? o : 1;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sv_stream_kernel<__nv_bfloat16, true>, NT, 0);
        d.occ[0][1] = o > 0 ? o : 1;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sv_stream_kernel<float, false>, NT, 0);
        d.occ[1][0] = o > 0 ? o : 1;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sv_stream_kernel<float, true>, NT, 0);
        d.occ[1][1] = o > 0 ? o : 1;
        const void *fin[2] = {(const void *)sv_finalize_kernel<__nv_bfloat16, true>,
                              (const void *)sv_finalize_kernel<float, true>};
        for (int i = 0; i < 2; ++i)
            if (cudaFuncSetAttribute(fin[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)RESCAN_SMEM_BYTES) != cudaSuccess)
                return nullptr;
        cudaGetLastError();
        d.sms = sms;
    }
    return &d;
}

// Split the flat range: as many CTAs as can be resident at once, but never fewer than E_MIN
// elements each; E is a multiple of 64 elements so that CTA boundaries stay 16-byte aligned.
static void plan_split(int64_t total, int resident, int64_t &E, int &G)
{
    int64_t g = resident;
    const int64_t by_min = (total + E_MIN - 1) / E_MIN;
    if (g > by_min) g = by_min;
    if (g > G_MAX) g = G_MAX;
    if (g < 1) g = 1;
    E = (total + g - 1) / g;
    E = (E + 63) / 64 * 64;
    G = (int)((total + E - 1) / E);
}

static int common_setup(Params &P, const void *logits, int dtype, int B, int rpr, int64_t V,
                        void *workspace, size_t ws_bytes, bool sample, int &occ_out)
{
    if (!logits || !workspace) return SPEC_VERIFY_EINVAL;
    if (dtype != SPEC_VERIFY_BF16 && dtype != SPEC_VERIFY_FP32) return SPEC_VERIFY_EINVAL;
    const int esize = dtype == SPEC_VERIFY_BF16 ? 2 : 4;
    if ((uintptr_t)logits % esize) return SPEC_VERIFY_EINVAL;
    if ((uintptr_t)workspace % 256) return SPEC_VERIFY_EWORKSPACE;
    const Layout L = layout(B, rpr, V);
    if (ws_bytes < L.total) return SPEC_VERIFY_EWORKSPACE;
    const DevInfo *d = device_info();
    if (!d) return SPEC_VERIFY_ECUDA;
    occ_out = d->occ[dtype == SPEC_VERIFY_FP32][sample ? 1 : 0];
    char *ws = static_cast<char *>(workspace);
    P.logits = logits;
    P.B = B;
    P.rpr = rpr;
    P.V = V;
    P.total = (int64_t)B * rpr * V;
    const int per_sm = (SV_CTAS_PER_SM > 0 && SV_CTAS_PER_SM < occ_out) ? SV_CTAS_PER_SM : occ_out;
    plan_split(P.total, d->sms * per_sm, P.E, P.G);
    P.mis = (int)(((uintptr_t)logits % 16) / esize);
    P.cnt1 = reinterpret_cast<unsigned *>(ws + L.cnt1);
    P.cnt2 = reinterpret_cast<unsigned *>(ws + L.cnt2);
    P.recs = reinterpret_cast<float2 *>(ws + L.recs);
    P.caps = reinterpret_cast<float *>(ws + L.caps);
    P.pend = reinterpret_cast<int4 *>(ws + L.pend);
    P.recs2 = reinterpret_cast<float2 *>(ws + L.recs2);
    P.C2 = residual_chunks(B, V);
    P.Ec2 = (V + P.C2 - 1) / P.C2;
    return SPEC_VERIFY_OK;
}

static void set_rng(Params &P, float temperature, uint64_t seed, uint64_t offset)
{
    P.cs = (float)(1.4426950408889634 / (double)temperature);
    P.key0 = (uint32_t)seed;
    P.key1 = (uint32_t)(seed >> 32);
    P.off0 = (uint32_t)offset;
    P.off1 = (uint32_t)(offset >> 32);
}

template <bool SAMPLE>
static int launch_stream(const Params &P, int dtype, cudaStream_t s)
{
    // The finaliser is launched as a programmatic dependent of the streaming kernel: its CTAs may
    // start early, stage the request's inputs, and wait (griddepcontrol) for the records.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P.B);
    cfg.blockDim = dim3(NT_FIN);
    cfg.dynamicSmemBytes = SAMPLE ? RESCAN_SMEM_BYTES : 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dtype == SPEC_VERIFY_BF16) {
        sv_stream_kernel<__nv_bfloat16, SAMPLE><<<P.G, NT, 0, s>>>(P);
        if (cudaGetLastError() != cudaSuccess) return SPEC_VERIFY_ECUDA;
        if (cudaLaunchKernelEx(&cfg, sv_finalize_kernel<__nv_bfloat16, SAMPLE>, P) != cudaSuccess)
            return SPEC_VERIFY_ECUDA;
    } else {
        sv_stream_kernel<float, SAMPLE><<<P.G, NT, 0, s>>>(P);
        if (cudaGetLastError() != cudaSuccess) return SPEC_VERIFY_ECUDA;
        if (cudaLaunchKernelEx(&cfg, sv_finalize_kernel<float, SAMPLE>, P) != cudaSuccess)
            return SPEC_VERIFY_ECUDA;
    }
    return cudaGetLastError() == cudaSuccess ? SPEC_VERIFY_OK : SPEC_VERIFY_ECUDA;
}

static bool temperature_ok(float t) { return t > 0.f && std::isfinite(t); }

}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_verify_workspace_bytes(int mode, int B, int k_or_N, int V)
{
    if (B < 1 || B > B_MAX || V < 1) return 0;
    int rpr;
    if (mode == SPEC_VERIFY_MODE_GREEDY || mode == SPEC_VERIFY_MODE_REJECTION) {
        if (k_or_N < 0 || k_or_N + 1 > MAX_RPR) return 0;
        rpr = k_or_N + 1;
    } else if (mode == SPEC_VERIFY_MODE_TREE) {
        if (k_or_N < 1 || k_or_N > MAX_RPR) return 0;
        rpr = k_or_N;
    } else {
        return 0;
    }
    return layout(B, rpr, V).total;
}

const char *spec_verify_strerror(int code)
{
    switch (code) {
    case SPEC_VERIFY_OK: return "ok";
    case SPEC_VERIFY_EINVAL: return "invalid argument";
    case SPEC_VERIFY_EWORKSPACE: return "workspace too small or not 256-byte aligned";
    case SPEC_VERIFY_ECUDA: return "CUDA launch or device query failed";
    case SPEC_VERIFY_ETOOBIG: return "the call needs more scratch than the built-in no-alloc buffer holds";
    case SPEC_VERIFY_DEV_BAD_TOKEN: return "device: a draft or node token outside [-1, V)";
    case SPEC_VERIFY_DEV_BAD_ROW: return "device: a logit row holds NaN or +inf, or no finite value";
    case SPEC_VERIFY_DEV_BAD_TREE: return "device: malformed tree (parents[0] != -1 or parents[j] outside [0, j))";
    case SPEC_VERIFY_DEV_DUP_SIBLING: return "device: two children of one node share a token";
    default: return "unknown status code";
    }
}

int spec_verify_greedy(const void *logits, int dtype, const int32_t *draft_ids, int B, int k,
                       int V, int32_t *out_tokens, int32_t *accept_len, void *workspace,
                       size_t ws_bytes, int32_t *dev_status, void *stream)
{
    if (B < 1 || B > B_MAX || k < 0 || k + 1 > MAX_RPR || V < 1) return SPEC_VERIFY_EINVAL;
    if ((k > 0 && !draft_ids) || !out_tokens || !accept_len) return SPEC_VERIFY_EINVAL;
    Params P;
    memset(&P, 0, sizeof P);
    int occ = 0;
    int rc = common_setup(P, logits, dtype, B, k + 1, V, workspace, ws_bytes, false, occ);
    if (rc) return rc;
    P.drafts = draft_ids;
    P.k = k;
    P.is_tree = 0;
    P.out_tokens = out_tokens;
    P.accept_len = accept_len;
    P.dev_status = dev_status;
    return launch_stream<false>(P, dtype, static_cast<cudaStream_t>(stream));
}

int spec_verify_rejection(const void *logits, int dtype, const int32_t *draft_ids,
                          const float *draft_probs, int B, int k, int V, float temperature,
                          uint64_t seed, uint64_t offset, int32_t *out_tokens,
                          int32_t *accept_len, float *out_probs, void *workspace,
                          size_t ws_bytes, int32_t *dev_status, void *stream)
{
    if (B < 1 || B > B_MAX || k < 0 || k + 1 > MAX_RPR || V < 1) return SPEC_VERIFY_EINVAL;
    if ((k > 0 && !draft_ids) || !out_tokens || !accept_len) return SPEC_VERIFY_EINVAL;
    if (!temperature_ok(temperature)) return SPEC_VERIFY_EINVAL;
    if (draft_probs && ((uintptr_t)draft_probs % 4)) return SPEC_VERIFY_EINVAL;
    Params P;
    memset(&P, 0, sizeof P);
    int occ = 0;
    int rc = common_setup(P, logits, dtype, B, k + 1, V, workspace, ws_bytes, true, occ);
    if (rc) return rc;
    P.drafts = draft_ids;
    P.q = (k > 0) ? draft_probs : nullptr;
    P.k = k;
    P.is_tree = 0;
    P.out_tokens = out_tokens;
    P.accept_len = accept_len;
    P.out_probs = out_probs;
    P.dev_status = dev_status;
    set_rng(P, temperature, seed, offset);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = launch_stream<true>(P, dtype, s);
    if (rc || !P.q) return rc;
    const unsigned grid = (unsigned)P.C2 * (unsigned)B;
    if (dtype == SPEC_VERIFY_BF16)
        sv_residual_kernel<__nv_bfloat16><<<grid, NT, 0, s>>>(P);
    else
        sv_residual_kernel<float><<<grid, NT, 0, s>>>(P);
    return cudaGetLastError() == cudaSuccess ? SPEC_VERIFY_OK : SPEC_VERIFY_ECUDA;
}

int spec_verify_tree(const void *logits, int dtype, const int32_t *node_tokens,
                     const int32_t *parents, int B, int N, int V, int mode, float temperature,
                     uint64_t seed, uint64_t offset, int32_t *out_tokens, int32_t *accept_index,
                     int32_t *accept_len, void *workspace, size_t ws_bytes, int32_t *dev_status,
                     void *stream)
{
    if (B < 1 || B > B_MAX || N < 1 || N > MAX_RPR || V < 1 || (mode != 0 && mode != 1))
        return SPEC_VERIFY_EINVAL;
    if (!node_tokens || !parents || !out_tokens || !accept_index || !accept_len) return SPEC_VERIFY_EINVAL;
    if (mode == 1 && !temperature_ok(temperature)) return SPEC_VERIFY_EINVAL;
    Params P;
    memset(&P, 0, sizeof P);
    int occ = 0;
    int rc = common_setup(P, logits, dtype, B, N, V, workspace, ws_bytes, mode == 1, occ);
    if (rc) return rc;
    P.node_tokens = node_tokens;
    P.parents = parents;
    P.k = N - 1;
    P.is_tree = 1;
    P.out_tokens = out_tokens;
    P.accept_index = accept_index;
    P.accept_len = accept_len;
    P.dev_status = dev_status;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (mode == 1) {
        set_rng(P, temperature, seed, offset);
        return launch_stream<true>(P, dtype, s);
    }
    return launch_stream<false>(P, dtype, s);
}

int spec_verify_philox(uint64_t seed, uint64_t offset, int n_slot, int n_req, uint32_t *out,
                       void *stream)
{
    if (n_slot < 1 || n_req < 1 || !out || (uintptr_t)out % 16) return SPEC_VERIFY_EINVAL;
    const int64_t n = (int64_t)n_slot * n_req;
    const int threads = 256;
    const int64_t blocks = (n + threads - 1) / threads;
    if (blocks > INT_MAX) return SPEC_VERIFY_EINVAL;
    sv_philox_kernel<<<(unsigned)blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        (uint32_t)seed, (uint32_t)(seed >> 32), (uint32_t)offset, (uint32_t)(offset >> 32), n_slot,
        n_req, out);
    return cudaGetLastError() == cudaSuccess ? SPEC_VERIFY_OK : SPEC_VERIFY_ECUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot allocate device memory at the point where they verify: code running
// inside a memory pool that forbids new allocations, an engine whose allocator is owned by
// another framework, or a host thread that must not take the driver's allocation lock.  For
// them, spec_verify_rejection_noalloc uses a scratch buffer that lives in this library's own
// device image instead of a caller-supplied workspace.  It is a fixed-size file-scope array, so
// every GPU that loads the library keeps SPEC_VERIFY_NOALLOC_SCRATCH_BYTES of it until the
// process exits.
// ---------------------------------------------------------------------------------------------
namespace sv {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_VERIFY_NOALLOC_SCRATCH_BYTES];

static std::mutex g_noalloc_mu;
static void *g_noalloc_ptr[64];

// The array's name is only a host-side stand-in; the device address is asked for once per
// device, with that device current.
static void *noalloc_scratch_address()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace sv

extern "C" int spec_verify_rejection_noalloc(const void *logits, int dtype,
                                             const int32_t *draft_ids, const float *draft_probs,
                                             int B, int k, int V, float temperature,
                                             uint64_t seed, uint64_t offset, int32_t *out_tokens,
                                             int32_t *accept_len, float *out_probs,
                                             int32_t *dev_status, void *stream)
{
    if (B < 1 || B > B_MAX || k < 0 || k + 1 > MAX_RPR || V < 1) return SPEC_VERIFY_EINVAL;
    const size_t need = spec_verify_workspace_bytes(SPEC_VERIFY_MODE_REJECTION, B, k, V);
    if (need == 0) return SPEC_VERIFY_EINVAL;
    if (need > SPEC_VERIFY_NOALLOC_SCRATCH_BYTES) return SPEC_VERIFY_ETOOBIG;
    void *scratch = noalloc_scratch_address();
    if (!scratch) return SPEC_VERIFY_ECUDA;
    // The scratch keeps whatever the previous call left; the arrival counters of the requests
    // this call uses must start at zero, so clear them (a memset, no allocation).
    const Layout L = layout(B, k + 1, V);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(scratch);
    if (cudaMemsetAsync(base + L.cnt1, 0, sizeof(unsigned) * (size_t)B, s) != cudaSuccess ||
        cudaMemsetAsync(base + L.cnt2, 0, sizeof(unsigned) * (size_t)B, s) != cudaSuccess)
        return SPEC_VERIFY_ECUDA;
    return spec_verify_rejection(logits, dtype, draft_ids, draft_probs, B, k, V, temperature, seed,
                                 offset, out_tokens, accept_len, out_probs, scratch,
                                 SPEC_VERIFY_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
