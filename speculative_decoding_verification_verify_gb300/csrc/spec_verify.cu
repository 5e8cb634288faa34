// spec_verify.cu -- the batched speculative-decoding verifier for GB300 (sm_103a), behind the
// C ABI declared in include/spec_verify.h.
//
// Hot path ("投机解码" [Speculative decoding], rustineverything, sections 目标模型怎么一次验证 and
// 接受规则为什么不改变分布; "The speculative decoding zoo", mlinterviewnotes 06-06, DFlash and
// verification-method sections):
//
//   sv_stream_kernel   -- one pass over all B * rows * V logits.  Each row is cut into chunks of
//                         CHUNK_VEC 16-byte vectors; one CTA per SM takes an equal run of the
//                         chunks, and its warps claim them one at a time from a shared counter,
//                         so every warp of an SM keeps streaming until the SM's run is done.  A
//                         warp folds its chunk into a (max, sum of 2^(l*cs - max*cs)) record,
//                         skipping the tokens that are children of the row's node (their logits
//                         are captured instead), or into an argmax record (greedy); a record
//                         carries the columns it covers.
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
#include "sv_decide.cuh"
#include "sv_stream.cuh"
#include "sv_rescan.cuh"
#include "sv_topkp.cuh"
#include "sv_topkp_ring.cuh"

#ifndef SV_PDL_TOPKP
#define SV_PDL_TOPKP 1
#endif
#ifndef SV_RESID_MINB
#define SV_RESID_MINB 4       // residual-kernel CTAs per SM the registers are budgeted for
#endif
#ifndef SV_RESID_TARGET
#define SV_RESID_TARGET 1024  // residual-kernel CTAs aimed at (column chunks per request x B)
#endif

namespace sv {

constexpr int NT_FIN_MAX = 256;  // threads of a finalising CTA: one warp per row, up to 8 rows
static_assert(NT_FIN_MAX == RESCAN_THREADS, "the stop row's rescan uses the whole finalising CTA");


// Per-request state of the finalising CTA.  Everything above the marked line depends only on the
// call's inputs and is staged before the streaming kernel's records are read.
struct FinSmem {
    int par[MAX_RPR], tok[MAX_RPR], dep[MAX_RPR];
    int first_child[MAX_RPR], next_sib[MAX_RPR];  // children with a usable token, by node index
    int ex_off[MAX_RPR], ex_n[MAX_RPR];           // each node's children, sorted by token column:
    int ex_col[MAX_RPR], ex_node[MAX_RPR];        //   ex_col/ex_node[ex_off[n] .. + ex_n[n])
    float qx[MAX_RPR], u[MAX_RPR], v[MAX_RPR];
    long long row_base[MAX_RPR];                  // first record index of each row
    int row_L[MAX_RPR];                           // records of each row
    // ---- from the records
    float row_mc[MAX_RPR], row_S[MAX_RPR];        // non-child mass S * 2^row_mc
    float row_M[MAX_RPR], row_tot[MAX_RPR];       // reference covering the children too; total in it
    float row_z[MAX_RPR];                         // non-child share of the row's mass
    float node_p[MAX_RPR];                        // p of node n's token in its parent's row
    float row_best[MAX_RPR];
    int row_arg[MAX_RPR];
    int cand[MAX_RPR];                            // the row's draw when it needs no rescan
    int rs_ok[MAX_RPR];                           // the row's draw rescans columns [rs_c0, rs_c1)
    int rs_c0[MAX_RPR], rs_c1[MAX_RPR];           //   of its crossing record,
    float rs_cum[MAX_RPR], rs_t[MAX_RPR];         //   mass before it, threshold (+inf: the last)
    RescanSmem RS;
    int path[MAX_RPR];
    int status;
    int stop;     // node at which the round stops
    int L;        // accepted drafts
    int mode;     // 0 emit argmax, 1 emit the stop row's draw, 2 residual pending
    int last_tok;
    float cs;     // the request's log2(e) / T
    float thr[MAX_RPR];  // each row's top-k / top-p logit threshold (-inf: not filtered)
};

// State of the residual kernel's last CTA.
struct ResidSmem {
    int rec;
    int take_last;
    int mode;
    float cum_before;
    float thresh;
    float z;
    DrawSmem D;
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
// Finalisation of request b: one warp per row merges the row's records, weighs the row's
// children and draws the row's candidate token; then one warp decides.
// ---------------------------------------------------------------------------------------------
constexpr int REC_PER_LANE = 4;  // records a lane keeps in registers for the draw's locate step

// Stage the request's structure, uniforms and record ranges (inputs only).
// VAR: the call has per-request temperatures or top-k / top-p thresholds (read from the staged
// F.cs / F.thr); without it the scale is the call's and nothing is filtered.
template <bool SAMPLE, bool VAR>
__device__ void stage_request(const Params &P, int b, FinSmem &F)
{
    const int tid = threadIdx.x, nt = blockDim.x;
    const int rpr = P.rpr;
    const int64_t V = P.V;
    const int64_t rbase = (int64_t)b * rpr;
    for (int n = tid; n < rpr; n += nt) {
        F.par[n] = n == 0 ? (P.is_tree && SV_INB(rbase, (int64_t)P.B * rpr, 301) ? __ldg(P.parents + rbase) : -1)
                          : node_parent(P, b, n);
        F.tok[n] = n == 0 ? -1 : node_token(P, b, n);
        float qv = 1.f;
        if (SAMPLE && P.q && n >= 1 && n <= P.k) {
            const int x = F.tok[n];
            const int64_t qi = ((int64_t)b * P.k + (n - 1)) * V + x;
            if (x >= 0 && (int64_t)x < V && SV_INB(qi, (int64_t)P.B * P.k * V, 302)) qv = __ldg(P.q + qi);
        }
        F.qx[n] = qv;
        if (VAR)
            F.thr[n] = (P.top_k || P.top_p) && SV_INB(rbase + n, (int64_t)P.B * rpr, 303) ? __ldcg(P.thr + rbase + n)
                                                                                          : NEG_INF;
        if (SAMPLE) {
            const float2 uv = uniforms(P, (uint32_t)n, (uint32_t)b);
            F.u[n] = uv.x;
            F.v[n] = uv.y;
        }
        const int64_t rr = rbase + n;
        F.row_base[n] = rr * P.nch;
        F.row_L[n] = (int)P.nch;
    }
    if (tid == 0) {
        F.status = 0;
        if (VAR) F.cs = P.temps && SV_INB(b, P.B, 304) ? cs_of(__ldg(P.temps + b)) : P.cs;
    }
    __syncthreads();
    if (!P.is_tree) {
        // A chain is a path: node n's only child is n + 1 (when its draft is usable).
        for (int n = tid; n < rpr; n += nt) {
            const int tk = F.tok[n];
            if (n >= 1 && (tk < -1 || (int64_t)tk >= V)) atomicMax(&F.status, SPEC_VERIFY_DEV_BAD_TOKEN);
            const bool has = n + 1 < rpr && F.tok[n + 1] >= 0 && (int64_t)F.tok[n + 1] < V;
            int off = 0;
            for (int m = 1; m <= n; ++m) off += (F.tok[m] >= 0 && (int64_t)F.tok[m] < V) ? 1 : 0;
            F.first_child[n] = has ? n + 1 : -1;
            F.next_sib[n] = -1;
            F.ex_n[n] = has ? 1 : 0;
            F.ex_off[n] = off;
            if (has) {
                F.ex_col[off] = F.tok[n + 1];
                F.ex_node[off] = n + 1;
            }
            F.dep[n] = n;
        }
        __syncthreads();
        return;
    }
    // Trees: validation (the largest fault code of the request wins), children and depths.
    for (int n = tid; n < rpr; n += nt) {
        int st = 0;
        const int tk = F.tok[n];
        if (n >= 1) {
            if (tk < -1 || (int64_t)tk >= V) st = SPEC_VERIFY_DEV_BAD_TOKEN;
            if (F.par[n] < 0 || F.par[n] >= n) st = max(st, SPEC_VERIFY_DEV_BAD_TREE);
            if (SAMPLE && tk >= 0) {
                for (int m = n + 1; m < rpr; ++m)
                    if (F.par[m] == F.par[n] && F.tok[m] == tk) st = max(st, SPEC_VERIFY_DEV_DUP_SIBLING);
            }
        } else if (F.par[0] != -1) {
            st = SPEC_VERIFY_DEV_BAD_TREE;
        }
        if (st) atomicMax(&F.status, st);
        int fc = -1, ns = -1, cnt = 0;
        for (int m = n + 1; m < rpr; ++m) {
            const bool usable = F.tok[m] >= 0 && (int64_t)F.tok[m] < V;
            if (usable && F.par[m] == n) {
                if (fc < 0) fc = m;
                ++cnt;
            }
            if (n >= 1 && ns < 0 && usable && F.par[m] == F.par[n]) ns = m;
        }
        F.first_child[n] = fc;
        F.next_sib[n] = ns;
        F.ex_n[n] = cnt;
        int d = 0, m = n;
        for (int it = 0; it < rpr && m > 0; ++it) {
            const int pa = F.par[m];
            if (pa < 0 || pa >= m) break;
            m = pa;
            ++d;
        }
        F.dep[n] = d;
    }
    __syncthreads();
    for (int n = tid; n < rpr; n += nt) {
        int off = 0;
        for (int m = 0; m < n; ++m) off += F.ex_n[m];
        F.ex_off[n] = off;
    }
    __syncthreads();
    // Each usable child takes its rank among its siblings by (token, node).
    for (int m = 1 + tid; m < rpr; m += nt) {
        const int pa = F.par[m], tk = F.tok[m];
        if (pa < 0 || pa >= m || tk < 0 || (int64_t)tk >= V) continue;
        int rank = 0;
        for (int s = pa + 1; s < rpr; ++s) {
            const int ts = F.tok[s];
            if (s != m && F.par[s] == pa && ts >= 0 && (int64_t)ts < V && (ts < tk || (ts == tk && s < m)))
                ++rank;
        }
        F.ex_col[F.ex_off[pa] + rank] = tk;
        F.ex_node[F.ex_off[pa] + rank] = m;
    }
    __syncthreads();
}

// What a warp keeps between merging a row's records and locating the draw's crossing in them.
struct RowState {
    float4 rr[REC_PER_LANE];  // a lane's contiguous run of q records (when inreg)
    float m[REC_PER_LANE];    // their masses in the reference mc (when inreg)
    float own, incl;          // the lane's run mass, and the running mass through it (when inreg)
    int64_t base;             // first record index of the row
    int L, q, off, cnt;       // records, records per lane, the row's children (ex_off, ex_n)
    bool inreg, bad;
    float mc, s, M, esum;     // non-child mass s * 2^mc; reference M covering the children too
};

// Row n of request b, by one warp, once the records are visible: merge the records, weigh the
// row's children.
template <typename T, bool SAMPLE, bool VAR>
__device__ void finish_row(const Params &P, int b, int n, FinSmem &F, int lane, RowState &rs)
{
    rs.base = F.row_base[n];
    rs.L = F.row_L[n];
    rs.bad = true;
    const int64_t base = rs.base;
    const int L = rs.L;
    if (!SAMPLE) {
        float best = NEG_INF;
        int idx = INT_MAX;
        for (int t = lane; t < L; t += 32) {
            if (!SV_INB(base + t, P.nchunks, 305)) continue;
            const float4 rec = __ldcg(P.recs + base + t);
            arg_merge(best, idx, rec.x, __float_as_int(rec.y));
        }
        warp_arg_merge(best, idx);
        if (lane == 0) {
            F.row_best[n] = best;
            F.row_arg[n] = idx;
            if (!(fabsf(best) < POS_INF)) atomicMax(&F.status, SPEC_VERIFY_DEV_BAD_ROW);
        }
        return;
    }
    // The children's captured logits and the row's records are loaded together.  Each lane takes
    // a contiguous run of q records; runs of up to REC_PER_LANE stay in registers for the draw's
    // locate step.
    const int off = F.ex_off[n], cnt = F.ex_n[n];
    rs.off = off;
    rs.cnt = cnt;
    float cap[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int e = lane + 32 * h;
        const int64_t ci = (int64_t)b * P.rpr + (e < cnt ? F.ex_node[off + e] : 0);
        cap[h] = e < cnt && SV_INB(ci, (int64_t)P.B * P.rpr, 306) ? __ldcg(P.caps + ci) : NEG_INF;
        if (VAR && !(cap[h] >= F.thr[n])) cap[h] = NEG_INF;  // below the row's top-k / top-p threshold
    }
    const int q = (L + 31) >> 5;
    rs.q = q;
    rs.inreg = q <= REC_PER_LANE;
    const float cs = VAR ? F.cs : P.cs;
    float mc = REF_NONE, s = 0.f, M, esum;
    float ec[2];
    if (rs.inreg) {
#pragma unroll
        for (int i = 0; i < REC_PER_LANE; ++i) {
            const int t = lane * q + i;
            rs.rr[i] = (i < q && t < L && SV_INB(base + t, P.nchunks, 307)) ? __ldcg(P.recs + base + t)
                                                                             : make_float4(REF_NONE, 0.f, 0.f, 0.f);
        }
        // The non-child reference mc (largest record reference) and the children's largest scaled
        // logit, reduced side by side; M covers both, so a child far above every other token
        // cannot overflow.
        float cm = fmaxf(cap[0] * cs, cap[1] * cs);
#pragma unroll
        for (int i = 0; i < REC_PER_LANE; ++i) mc = fmaxf(mc, rs.rr[i].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
            cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
        }
        M = fmaxf(mc, cm);
        // Each record's mass in the reference mc (kept for the draw's locate step), the children's
        // weights in M; the two sums and the running sum over the lanes' runs, side by side.
        float own = 0.f;
#pragma unroll
        for (int i = 0; i < REC_PER_LANE; ++i) {
            rs.m[i] = (rs.rr[i].y == 0.f) ? 0.f : rs.rr[i].y * ex2(rs.rr[i].x - mc);
            own += rs.m[i];
        }
        float le = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            ec[h] = (lane + 32 * h < cnt) ? ex2(fmaf(cap[h], cs, -M)) : 0.f;
            le += ec[h];
        }
        float incl = own;
        s = own;
        esum = le;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            s += __shfl_xor_sync(0xffffffffu, s, o);
            esum += __shfl_xor_sync(0xffffffffu, esum, o);
            if (lane >= o) incl += y;
        }
        rs.own = own;
        rs.incl = incl;
    } else {
        for (int t = lane; t < L; t += 32) {
            if (!SV_INB(base + t, P.nchunks, 308)) continue;
            const float4 rec = __ldcg(P.recs + base + t);
            rec_merge(mc, s, rec.x, rec.y);
        }
        warp_rec_merge(mc, s);
        M = mc;
#pragma unroll
        for (int h = 0; h < 2; ++h) M = fmaxf(M, cap[h] * cs);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        esum = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            ec[h] = (lane + 32 * h < cnt) ? ex2(fmaf(cap[h], cs, -M)) : 0.f;
            esum += ec[h];
        }
        esum = warp_sum(esum);
    }
    const float s_ref = (s == 0.f) ? 0.f : s * ex2(mc - M);
    const float tot = s_ref + esum;
#pragma unroll
    for (int h = 0; h < 2; ++h)
        if (lane + 32 * h < cnt) F.node_p[F.ex_node[off + lane + 32 * h]] = ec[h] / tot;
    const bool bad = !(s >= 0.f) || !(s < POS_INF) || !(tot > 0.f) || !(tot < POS_INF);
    rs.bad = bad;
    rs.mc = mc;
    rs.s = s;
    rs.M = M;
    rs.esum = esum;
    if (lane == 0) {
        F.row_mc[n] = mc;
        F.row_S[n] = s;
        F.row_M[n] = M;
        F.row_tot[n] = tot;
        F.row_z[n] = s_ref / tot;
        F.cand[n] = -1;
        F.rs_ok[n] = 0;
        if (bad) atomicMax(&F.status, SPEC_VERIFY_DEV_BAD_ROW);
    }
}

// The row's draw, children excluded, threshold v * Z with Z the non-child mass: locate the
// record holding the crossing (F.rs_*) for the rescan, or, when every non-child token is -inf,
// draw among the children directly (F.cand).
template <bool VAR>
__device__ void row_draw_prep(const Params &P, int b, int n, FinSmem &F, int lane, const RowState &rs)
{
    const float vdraw = F.v[P.is_tree ? F.dep[n] : n];
    const float s = rs.s, mc = rs.mc;
    const int L = rs.L, q = rs.q;
    if (s > 0.f) {
        const float t = vdraw * s;
        int fi = -1;         // crossing record (relative to the row's first), or the last positive
        float before = 0.f;  // mass of the row's records before it
        bool take_last = false;
        float4 frec = make_float4(0.f, 0.f, 0.f, 0.f);
        if (rs.inreg) {
            const float own = rs.own, incl = rs.incl;
            const float(&m)[REC_PER_LANE] = rs.m;
            float excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (lane == 0) excl = 0.f;
            const unsigned hit = __ballot_sync(0xffffffffu, excl + own > t);
            const unsigned pos = __ballot_sync(0xffffffffu, own > 0.f);
            take_last = hit == 0;
            const int who = take_last ? 31 - __clz(pos) : __ffs(hit) - 1;
            if (pos && lane == who) {
                float c = excl, lpc = 0.f;
                int lpi = -1;
#pragma unroll
                for (int i = 0; i < REC_PER_LANE; ++i) {
                    if (m[i] > 0.f) {
                        if (fi < 0 && !take_last && c + m[i] > t) {
                            fi = i;
                            before = c;
                        }
                        if (fi < 0) {
                            lpi = i;
                            lpc = c;
                        }
                    }
                    c += m[i];
                }
                if (fi < 0) {  // take_last, or rounding: the run crossed, its records did not
                    fi = lpi;
                    before = lpc;
                    take_last = true;
                }
#pragma unroll
                for (int i = 0; i < REC_PER_LANE; ++i)
                    if (i == fi) frec = rs.rr[i];
                fi += lane * q;
            }
        } else {
            Locate Lc;
            for (int c0 = 0; c0 < L; c0 += 32) {
                const float4 rec = c0 + lane < L && SV_INB(rs.base + c0 + lane, P.nchunks, 309)
                                       ? __ldcg(P.recs + rs.base + c0 + lane)
                                       : make_float4(REF_NONE, 0.f, 0.f, 0.f);
                if (locate_chunk(Lc, rec_mass(rec, mc), c0, t, lane)) break;
            }
            if (lane == 0) {
                fi = Lc.found >= 0 ? Lc.found : Lc.lastpos;
                before = Lc.found >= 0 ? Lc.before : Lc.lp_before;
                take_last = Lc.found < 0;
                if (fi >= 0 && SV_INB(rs.base + fi, P.nchunks, 310)) frec = __ldcg(P.recs + rs.base + fi);
            }
        }
        if (fi >= 0) {  // exactly one lane holds it
            F.rs_c0[n] = __float_as_int(frec.z);
            F.rs_c1[n] = __float_as_int(frec.w);
            F.rs_cum[n] = before;
            F.rs_t[n] = take_last ? POS_INF : t;
            F.rs_ok[n] = 1;
        }
    } else if (lane == 0) {
        // Every non-child token is -inf: draw among the children by p, in column order.
        const float t = vdraw * rs.esum;
        float c = 0.f;
        int lastc = -1, drawn = -1;
        for (int e = 0; e < rs.cnt && drawn < 0; ++e) {
            const int64_t ci = (int64_t)b * P.rpr + F.ex_node[rs.off + e];
            const float cp = SV_INB(ci, (int64_t)P.B * P.rpr, 311) ? __ldcg(P.caps + ci) : NEG_INF;
            const float w = (!VAR || cp >= F.thr[n]) ? ex2(fmaf(cp, VAR ? F.cs : P.cs, -rs.M)) : 0.f;
            if (w > 0.f) {
                lastc = F.ex_col[rs.off + e];
                c += w;
                if (c > t) drawn = lastc;
            }
        }
        F.cand[n] = drawn >= 0 ? drawn : lastc;
    }
}

template <typename T, bool SAMPLE, bool VAR>
__device__ void finalize_request(const Params &P, int b, FinSmem &F)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwf = blockDim.x >> 5;
    const int rpr = P.rpr;

    stage_request<SAMPLE, VAR>(P, b, F);
    // From here on the streaming kernel's records and captures are read.
    pdl_wait();
    // Each warp merges its rows and, when sampling, locates each row's crossing record at once:
    // whichever row the decision stops at, its draw needs only the rescan of that record.
    RowState rs;
    for (int n = warp; n < rpr; n += nwf) {
        finish_row<T, SAMPLE, VAR>(P, b, n, F, lane, rs);
        if (SAMPLE && !rs.bad) row_draw_prep<VAR>(P, b, n, F, lane, rs);
    }
    __syncthreads();
    // A plain chain's decision is a few shared-memory reads and a ballot: every warp takes it
    // itself.  Block verification and trees decide in warp 0.
    const bool chain = !P.is_tree && !P.block;
    int L = 0, stop = 0, mode = 0;
    if (chain) {
        if (F.status == 0) {
            L = stop = chain_stop<SAMPLE, VAR>(P, F, lane);
            mode = chain_mode<SAMPLE>(P, F, stop);
        }
    } else {
        if (warp == 0 && !(P.block && P.q)) decide_request<SAMPLE, VAR>(P, F, lane);
        __syncthreads();
        L = F.L;
        stop = F.stop;
        mode = F.mode;
    }
    const bool faulted = F.status != 0;

    if (SAMPLE && P.block && P.q) {
        // Block verification with draft probabilities: the residual masses need every row's
        // statistics, so the block kernel decides and draws.  Hand it each present row's
        // reference, total and prefix weight w_L = min(1, w_{L-1} p(x)/q(x)).
        if (faulted) {
            for (int i = tid; i <= P.k; i += blockDim.x)
                if (SV_INB((int64_t)b * (P.k + 1) + i, (int64_t)P.B * (P.k + 1), 320))
                    P.out_tokens[(int64_t)b * (P.k + 1) + i] = -1;
            if (tid == 0 && SV_INB(b, P.B, 321)) {
                P.accept_len[b] = -1;
                raise_status(P.dev_status, F.status);
                P.pend[b] = make_int4(-1, 0, 0, 0);
            }
            return;
        }
        if (tid == 0) {
            int ke = P.k;
            for (int i = 0; i < P.k; ++i)
                if (F.tok[i + 1] < 0) {
                    ke = i;
                    break;
                }
            float w = 1.f;
            for (int L = 0; L <= ke; ++L) {
                if (SV_INB((int64_t)b * rpr + L, (int64_t)P.B * rpr, 322))
                    P.bpend[(int64_t)b * rpr + L] = make_float4(F.row_M[L], F.row_tot[L], w, 1.f);
                if (L < ke) {
                    const float px = F.node_p[L + 1], qx = F.qx[L + 1];
                    w = (w * px <= 0.f) ? 0.f : (qx <= 0.f ? 1.f : fminf(1.f, w * px / qx));
                }
            }
            if (SV_INB(b, P.B, 323)) P.pend[b] = make_int4(ke, 0, 0, 1);
        }
        return;
    }

    // Outputs.
    const int out_w = P.is_tree ? rpr : P.k + 1;
    int32_t *ot = P.out_tokens + (int64_t)b * out_w;
    [[maybe_unused]] const int64_t ot_n = (int64_t)P.B * out_w;  // extents for debug builds' range checks
    [[maybe_unused]] const int64_t op_n = (int64_t)P.B * (P.k + 1) * 3;
    if (faulted) {
        for (int i = tid; i < out_w; i += blockDim.x) {
            if (SV_INB((int64_t)b * out_w + i, ot_n, 324)) ot[i] = -1;
            if (P.is_tree && SV_INB((int64_t)b * rpr + i, ot_n, 325)) P.accept_index[(int64_t)b * rpr + i] = -1;
        }
        if (tid == 0 && SV_INB(b, P.B, 326)) {
            P.accept_len[b] = -1;
            raise_status(P.dev_status, F.status);
        }
        if (P.out_probs && !P.is_tree)
            for (int i = tid; i < (P.k + 1) * 3; i += blockDim.x)
                if (SV_INB((int64_t)b * (P.k + 1) * 3 + i, op_n, 327)) P.out_probs[(int64_t)b * (P.k + 1) * 3 + i] = 0.f;
        if (P.q && !P.is_tree && tid == 0 && SV_INB(b, P.B, 328)) P.pend[b] = make_int4(-1, 0, 0, 0);
        return;
    }
    int last = -1;
    if (mode == 0) {
        last = F.row_arg[stop];
    } else if (SAMPLE && mode == 1) {
        // The draw at the stop row: the whole CTA rescans the columns of its crossing record.
        int drawn = F.cand[stop];
        if (F.rs_ok[stop]) {
            const int64_t r = (int64_t)b * rpr + stop;
            const T *row = reinterpret_cast<const T *>(P.logits) + r * P.V;
            uint4 w[RESCAN_ROUNDS];
            if (!(SV_INB(F.rs_c0[stop], P.V + 1, 341) && SV_INB(F.rs_c1[stop], P.V + 1, 342))) F.rs_c1[stop] = F.rs_c0[stop];
            load_range<T>(row, r * P.V, P.total, P.mis, F.rs_c0[stop], F.rs_c1[stop], w);
            drawn = rescan_range<T, VAR>(r * P.V, P.mis, F.rs_c0[stop], F.rs_c1[stop], VAR ? F.cs : P.cs,
                                         F.row_mc[stop], VAR ? F.thr[stop] : NEG_INF, F.rs_t[stop], F.rs_cum[stop],
                                         F.ex_col + F.ex_off[stop], F.ex_n[stop], w, F.RS);
        }
        last = drawn >= 0 ? drawn : 0;  // < 0 only through rounding
    }
    for (int i = tid; i < out_w; i += blockDim.x) {
        int v = -1;
        if (i < L) v = F.tok[P.is_tree ? F.path[i] : i + 1];
        else if (i == L) v = last;
        if (SV_INB((int64_t)b * out_w + i, ot_n, 329)) ot[i] = v;
        if (P.is_tree && SV_INB((int64_t)b * rpr + i, ot_n, 330))
            P.accept_index[(int64_t)b * rpr + i] = (i == 0) ? 0 : (i <= L ? F.path[i - 1] : -1);
    }
    if (!SAMPLE && P.out_probs && !P.is_tree)  // a greedy request of a mixed batch
        for (int i = tid; i < (P.k + 1) * 3; i += blockDim.x)
            if (SV_INB((int64_t)b * (P.k + 1) * 3 + i, op_n, 331)) P.out_probs[(int64_t)b * (P.k + 1) * 3 + i] = 0.f;
    if (tid == 0 && SV_INB(b, P.B, 332)) {
        P.accept_len[b] = L;
        if (!SAMPLE && P.q && !P.is_tree) P.pend[b] = make_int4(-1, 0, 0, 0);
        if (SAMPLE && P.q && !P.is_tree) {
            if (mode == 2)
                P.pend[b] = make_int4(stop, __float_as_int(F.row_M[stop]), __float_as_int(F.row_tot[stop]), 1);
            else
                P.pend[b] = make_int4(-1, 0, 0, 0);
        }
    }
    if (SAMPLE && P.out_probs && !P.is_tree) {
        float *op = P.out_probs + (int64_t)b * (P.k + 1) * 3;
        for (int i = tid; i <= P.k; i += blockDim.x) {
            float p0 = 0.f, q0 = 0.f, z = 0.f;
            if (i < P.k && F.tok[i + 1] >= 0) {
                p0 = F.node_p[i + 1];
                q0 = F.qx[i + 1];
            }
            if (i == stop && mode == 1) z = F.row_z[i];
            if (!SV_INB((int64_t)b * (P.k + 1) * 3 + 3 * i + 2, op_n, 333)) continue;
            op[3 * i + 0] = p0;
            op[3 * i + 1] = q0;
            op[3 * i + 2] = z;
        }
    }
}

// ---------------------------------------------------------------------------------------------
// The streaming kernel: every CTA folds its share of the flat logits range into per-warp records.
// ---------------------------------------------------------------------------------------------
// KIND: 0 greedy, 1 sampling, 2 a temperature per request (greedy or sampling per chunk),
// 3 as 2 with each row's top-k / top-p threshold applied in the sampling fold, 4 sampling at one
// temperature with each row's threshold (the sampling fold alone: 24 warps, as kinds 0 and 1).
template <typename T, int KIND>
__global__ void __launch_bounds__(stream_threads(KIND), 1) sv_stream_kernel(const Params P)
{
    constexpr bool SAMPLE = KIND != 0;
    __shared__ unsigned next_chunk;
    constexpr int VEC = Elt<T>::VEC;
    const int g = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    pdl_launch_dependents();
    const int64_t q0 = (int64_t)g * P.cpc;
    const int64_t nq = min(q0 + P.cpc, P.nchunks) - q0;
    if (tid == 0) next_chunk = 0;
    __syncthreads();
    // Claims run one chunk ahead, so the shared-memory atomic is off the critical path.
    unsigned c = 0;
    if (lane == 0) c = atomicAdd(&next_chunk, 1u);
    c = __shfl_sync(0xffffffffu, c, 0);
    int cur_b = -1, cur_n = -1;
    NodeView nv;
    Kids kd;
    kd.col[0] = kd.col[1] = INT_MAX;
    float cs = P.cs;
    float thr = NEG_INF;
    bool greedy_b = false;
    // A warp's claims only grow, by about a round of claims at a time, so its chunk's row (and the
    // row's request and node) are advanced from the last claim's instead of divided out afresh.
    int64_t r = -1, rq = 0;  // the row, and its first chunk's index
    int b = 0, n = -1;       // its request and node (rows < 2^31)
    while ((int64_t)c < nq) {
        unsigned nxt = 0;
        if (lane == 0) nxt = atomicAdd(&next_chunk, 1u);
        const int64_t q = q0 + c;
        if (r < 0 || q - rq >= 4 * P.nch) {
            r = q / P.nch;
            rq = r * P.nch;
            b = (int)(r / P.rpr);
            n = (int)(r - (int64_t)b * P.rpr);
        }
        while (q - rq >= P.nch) {
            ++r;
            rq += P.nch;
            if (++n == P.rpr) {
                n = 0;
                ++b;
            }
        }
        const int64_t j = q - rq;
        const Seg sg = chunk_of<VEC>(P, r, j);
        const T *row = reinterpret_cast<const T *>(P.logits) + r * P.V;
        float *caps = P.caps + (int64_t)b * P.rpr;
        const bool rec_ok = SV_INB(q, P.nchunks, 205);
        if (KIND == 2 || KIND == 3) {
            // The request's temperature decides the chunk's fold; nodes, children and the row's
            // threshold are refreshed first (global loads only when the request or row changes).
            if (b != cur_b || n != cur_n) {
                if (b != cur_b) {
                    load_nodes(P, b, lane, nv);
                    const float Tb = P.temps && SV_INB(b, P.B, 206) ? __ldg(P.temps + b) : 1.f;
                    greedy_b = Tb == 0.f;
                    cs = greedy_b ? 1.f : (P.temps ? cs_of(Tb) : P.cs);
                }
                kids_of(P, nv, n, kd);
                if (KIND == 3) thr = SV_INB(r, (int64_t)P.B * P.rpr, 207) ? __ldcg(P.thr + r) : NEG_INF;
                cur_b = b;
                cur_n = n;
            }
            if (greedy_b)
                stream_chunk<T, false, false>(row, sg, lane, cs, kd, caps, P.recs + q, []() {}, thr, r * P.V, P.total,
                                              P.rpr, rec_ok);
            else
                stream_chunk<T, true, KIND == 3>(row, sg, lane, cs, kd, caps, P.recs + q, []() {}, thr, r * P.V,
                                                 P.total, P.rpr, rec_ok);
        } else if (KIND == 4) {
            // The row's children and threshold are refreshed when the row changes.
            if (b != cur_b || n != cur_n) {
                if (b != cur_b) load_nodes(P, b, lane, nv);
                kids_of(P, nv, n, kd);
                thr = SV_INB(r, (int64_t)P.B * P.rpr, 207) ? __ldcg(P.thr + r) : NEG_INF;
                cur_b = b;
                cur_n = n;
            }
            stream_chunk<T, true, true>(row, sg, lane, cs, kd, caps, P.recs + q, []() {}, thr, r * P.V, P.total,
                                        P.rpr, rec_ok);
        } else {
            // The row's child tokens are (re)derived while the chunk's first loads are in flight.
            stream_chunk<T, SAMPLE, false>(row, sg, lane, cs, kd, caps, P.recs + q, [&]() {
                if (SAMPLE && (b != cur_b || n != cur_n)) {
                    if (b != cur_b) load_nodes(P, b, lane, nv);
                    kids_of(P, nv, n, kd);
                    cur_b = b;
                    cur_n = n;
                }
            }, NEG_INF, r * P.V, P.total, P.rpr, rec_ok);
        }
        c = __shfl_sync(0xffffffffu, nxt, 0);
    }
}

// ---------------------------------------------------------------------------------------------
// The finalising kernel: one CTA per request merges its records, decides and draws.
// ---------------------------------------------------------------------------------------------
// VAR: per-request temperatures (a greedy request, T = 0, takes the argmax path) or top-k /
// top-p thresholds; a separate instantiation, so the plain kernels carry only their own code.
template <typename T, bool SAMPLE, bool VAR>
__global__ void __launch_bounds__(NT_FIN_MAX) sv_finalize_kernel(const Params P)
{
    __shared__ FinSmem F;
    const int b = (int)blockIdx.x;
    if (VAR && P.temps && SV_INB(b, P.B, 340) && __ldg(P.temps + b) == 0.f) finalize_request<T, false, false>(P, b, F);
    else finalize_request<T, SAMPLE, VAR>(P, b, F);
}

// 8 consecutive logits (one 16-byte vector of bf16, two of fp32) or q values, as floats; the
// address must be 16-byte aligned.
template <typename T>
__device__ __forceinline__ void load8(const T *p, float (&x)[8])
{
    if (sizeof(T) == 2) {
        float y[8];
        Elt<__nv_bfloat16>::unpack(ldg_stream(p), y);
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = y[j];
    } else {
        const uint4 a = ldg_stream(p), c = ldg_stream(p + 4);
        x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
        x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
        x[4] = __uint_as_float(c.x); x[5] = __uint_as_float(c.y);
        x[6] = __uint_as_float(c.z); x[7] = __uint_as_float(c.w);
    }
}

// One warp's residual sums over the columns [w0, w1) of a logit row: zr += max(0, w p - q) and
// zp += p, with p = 2^(l cs - mc) * inv (0 for logits below thr when FILT) and q = 0 without a
// q row.  lflat / qflat are the row's first element in the flat logits / q arrays, whose bases
// are lmis / qmis elements past a 16-byte boundary.  Groups of 8 columns whose logits and q both
// start on a 16-byte boundary are read with 16-byte loads, RESID_GROUPS groups per lane in flight; the
// columns before the first group and after the last (fewer than 8 each), or the whole span
// when the logits and the q row cannot be aligned at the same column, are read one by one.
template <typename T, bool FILT>
__device__ __forceinline__ void resid_sums(const T *row, const float *qrow, int64_t lflat, int64_t qflat,
                                           int lmis, int qmis, int64_t w0, int64_t w1, float cs, float mc,
                                           float inv, float w, float thr, int lane, float &zr, float &zp)
{
    constexpr int VEC = Elt<T>::VEC;
    auto add = [&](float l, float q) {
        const float p = (!FILT || l >= thr) ? ex2(fmaf(l, cs, -mc)) * inv : 0.f;
        zp += p;
        zr += fmaxf(0.f, w * p - q);
    };
    // Logits start a vector at the columns congruent to h (mod VEC); q (4 floats to a vector) at
    // those congruent to h mod 4 either everywhere or nowhere, as VEC is 4 or 8.
    int64_t h = w0 + (VEC - (int)((lmis + lflat + w0) % VEC)) % VEC;
    const bool vec_ok = qmis >= 0 && (!qrow || (qmis + qflat + h) % 4 == 0);
    if (!vec_ok || h > w1) h = w1;
    const int64_t ng = (w1 - h) / 8, t0 = h + ng * 8;
    for (int64_t c = w0 + lane; c < h; c += 32) add(Elt<T>::load(row, c), qrow ? __ldg(qrow + c) : 0.f);
    for (int64_t g0 = lane; g0 < ng; g0 += 32 * RESID_GROUPS) {
        float l[RESID_GROUPS][8], q[RESID_GROUPS][8];
#pragma unroll
        for (int u = 0; u < RESID_GROUPS; ++u) {
            const int64_t g = g0 + 32 * u;
            if (g < ng) {
                load8<T>(row + h + g * 8, l[u]);
                if (qrow) load8<float>(qrow + h + g * 8, q[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < RESID_GROUPS; ++u) {
            if (g0 + 32 * u >= ng) break;
#pragma unroll
            for (int j = 0; j < 8; ++j) add(l[u][j], qrow ? q[u][j] : 0.f);
        }
    }
    for (int64_t c = t0 + lane; c < w1; c += 32) add(Elt<T>::load(row, c), qrow ? __ldg(qrow + c) : 0.f);
}

// Elements the q array's base lies past a 16-byte boundary, or -1 when it is not 4-byte aligned.
__device__ __forceinline__ int q_mis(const float *q)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(q);
    return (a & 3) ? -1 : (int)((a & 15) >> 2);
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
    int use_p;           // draw from p instead (residual mass underflowed, or no draft here)
    float w;             // prefix weight of block verification (1 for the standard residual)
    float thr;           // the row's top-k / top-p threshold: logits below it have p = 0
    __device__ Raw prefetch(int64_t gi) const
    {
        Raw r;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t c = col0 + gi * 8 + j;
            const bool in = c < col1;
            r.l[j] = in ? Elt<T>::load(row, c) : NEG_INF;
            r.q[j] = (in && qrow) ? __ldg(qrow + c) : 0.f;
        }
        return r;
    }
    __device__ int weights(const Raw &r, int64_t gi, float (&w)[8]) const
    {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float p = r.l[j] >= thr ? ex2(fmaf(r.l[j], cs, -mc)) * inv : 0.f;
            w[j] = use_p ? p : fmaxf(0.f, this->w * p - r.q[j]);
        }
        return (int)(col0 + gi * 8);
    }
};

template <typename T>
__global__ void __launch_bounds__(NT, SV_RESID_MINB) sv_residual_kernel(const Params P)
{
    __shared__ ResidSmem F;
    __shared__ int is_last;
    const int c = (int)(blockIdx.x % (unsigned)P.C2), b = (int)(blockIdx.x / (unsigned)P.C2);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (!SV_INB(b, P.B, 501)) return;
    const int4 pd = P.pend[b];
    if (pd.w != 1) return;
    const int j = pd.x;
    const float mc = __int_as_float(pd.y), tot = __int_as_float(pd.z);
    const float inv = 1.f / tot;
    const float cs = P.temps ? cs_of(__ldg(P.temps + b)) : P.cs;
    const int64_t V = P.V;
    const int64_t r = (int64_t)b * P.rpr + j;
    if (!SV_INB(j, P.k, 502)) return;  // a pending residual draw sits at a draft slot
    const float thr = P.thr && (P.top_k || P.top_p) ? __ldcg(P.thr + r) : NEG_INF;
    const void *row = reinterpret_cast<const T *>(P.logits) + r * V;
    const float *qrow = P.q + ((int64_t)b * P.k + j) * V;
    const int64_t cc0 = (int64_t)c * P.Ec2, cc1 = min(cc0 + P.Ec2, V);
    const int64_t span = (cc1 - cc0 + NW - 1) / NW;
    const int64_t w0 = min(cc0 + warp * span, cc1), w1 = min(w0 + span, cc1);
    float zr = 0.f, zp = 0.f;
    // The warp's columns [w0, w1) of the row and of its q row: both ends in range.
    if (w1 <= w0 || (SV_INB(r * V + w1 - 1, P.total, 503) && SV_INB(((int64_t)b * P.k + j) * V + w1 - 1,
                                                                     (int64_t)P.B * P.k * V, 504)))
        resid_sums<T, true>(reinterpret_cast<const T *>(row), qrow, r * V, ((int64_t)b * P.k + j) * V, P.mis,
                            q_mis(P.q), w0, w1, cs, mc, inv, 1.f, thr, lane, zr, zp);
    zr = warp_sum(zr);
    zp = warp_sum(zp);
    const int64_t ri = ((int64_t)b * P.C2 + c) * NW + warp;
    if (lane == 0 && SV_INB(ri, (int64_t)P.B * P.C2 * NW, 505)) P.recs2[ri] = make_float2(zr, zp);
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
    if (!SV_INB((int64_t)b * P.C2 * NW + L - 1, (int64_t)P.B * P.C2 * NW, 506)) return;
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
            F.z = use_p ? 1.f : zr_t;
        }
    }
    __syncthreads();
    int drawn = -1;
    if (F.rec >= 0) {
        const int rc = F.rec / NW, rw = F.rec % NW;
        const int64_t a0 = (int64_t)rc * P.Ec2, a1 = min(a0 + P.Ec2, V);
        const int64_t sp = (a1 - a0 + NW - 1) / NW;
        const int64_t s0 = min(a0 + rw * sp, a1), s1 = SV_INB(min(s0 + sp, a1) - 1, V, 507) ? min(s0 + sp, a1) : s0;
        ResidSrc<T> src{row, qrow, s0, s1, cs, mc, inv, F.mode, 1.f, thr};
        draw_init(F.D, F.cum_before);
        draw_span<2>(src, (s1 - s0 + 7) / 8, F.take_last ? POS_INF : F.thresh, F.D);
        drawn = F.D.found >= 0 ? F.D.found : F.D.lastpos;
    }
    if (tid == 0) {
        if (SV_INB((int64_t)b * (P.k + 1) + j, (int64_t)P.B * (P.k + 1), 508))
            P.out_tokens[(int64_t)b * (P.k + 1) + j] = drawn >= 0 ? drawn : 0;
        if (P.out_probs && SV_INB(((int64_t)b * (P.k + 1) + j) * 3 + 2, (int64_t)P.B * (P.k + 1) * 3, 509))
            P.out_probs[((int64_t)b * (P.k + 1) + j) * 3 + 2] = F.z;
        P.cnt2[b] = 0u;
    }
}

// ---------------------------------------------------------------------------------------------
// Block verification with draft probabilities ("The speculative decoding zoo", block branch of
// the rejection sampler, after Sun et al.).  Grid (C2 chunks, rows, B): each CTA sums, over its
// chunk of row L, the residual max(0, w_L p - q) and p per warp.  The last CTA of a request
// (atomic arrival counter, nothing waits) forms r_L, the tests h_L = r_L / (r_L + 1 - w_L)
// (h = w at the last present draft), takes the largest passing length j, and draws the next
// token from max(0, w_j p_j - q_j) (from p_j at the last present draft) by locating the
// crossing warp record and rescanning that part of the row.
// ---------------------------------------------------------------------------------------------
struct BlockSmem {
    float r[MAX_RPR], z[MAX_RPR];  // per row: residual mass, p mass
    int j;
    int use_p;
    float Z, t;
    ResidSmem R;
};

template <typename T>
__global__ void __launch_bounds__(NT, 4) sv_block_kernel(const Params P)
{
    __shared__ BlockSmem S;
    __shared__ int is_last;
    const int rpr = P.rpr;
    const int c = (int)(blockIdx.x % (unsigned)P.C2);
    const int rest = (int)(blockIdx.x / (unsigned)P.C2);
    const int L = rest % rpr, b = rest / rpr;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (!SV_INB(b, P.B, 601)) return;
    const int4 pd = P.pend[b];
    if (pd.w != 1) return;
    const int ke = pd.x;
    if (L > ke || !SV_INB(ke, rpr, 602)) return;
    const int64_t V = P.V;
    {
        const float4 bp = P.bpend[(int64_t)b * rpr + L];
        const float mc = bp.x, inv = 1.f / bp.y, w = bp.z;
        const int64_t r = (int64_t)b * rpr + L;
        const void *row = reinterpret_cast<const T *>(P.logits) + r * V;
        const float *qrow = L < P.k ? P.q + ((int64_t)b * P.k + L) * V : nullptr;
        const int64_t cc0 = (int64_t)c * P.Ec2, cc1 = min(cc0 + P.Ec2, V);
        const int64_t span = (cc1 - cc0 + NW - 1) / NW;
        const int64_t w0 = min(cc0 + warp * span, cc1), w1 = min(w0 + span, cc1);
        float zr = 0.f, zp = 0.f;
        if (w1 <= w0 || (SV_INB(r * V + w1 - 1, P.total, 603) &&
                         (!qrow || SV_INB(((int64_t)b * P.k + L) * V + w1 - 1, (int64_t)P.B * P.k * V, 604))))
            resid_sums<T, false>(reinterpret_cast<const T *>(row), qrow, r * V, ((int64_t)b * P.k + L) * V, P.mis,
                                 q_mis(P.q), w0, w1, P.cs, mc, inv, w, NEG_INF, lane, zr, zp);
        zr = warp_sum(zr);
        zp = warp_sum(zp);
        if (lane == 0 && SV_INB((r * P.C2 + c) * NW + warp, (int64_t)P.B * rpr * P.C2 * NW, 605))
            P.recs3[(r * P.C2 + c) * NW + warp] = make_float2(zr, zp);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned old = atomicAdd(P.cnt2 + b, 1u);
        is_last = (old == (unsigned)((ke + 1) * P.C2) - 1u);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    // Last CTA of request b: row masses, the decision, then the draw.
    const int per_row = P.C2 * NW;
    if (!SV_INB(((int64_t)b * rpr + ke) * per_row + per_row - 1, (int64_t)P.B * rpr * per_row, 606)) return;
    for (int Lr = warp; Lr <= ke; Lr += NW) {
        const float2 *rb = P.recs3 + ((int64_t)b * rpr + Lr) * per_row;
        float a = 0.f, z = 0.f;
        for (int t = lane; t < per_row; t += 32) {
            const float2 x = __ldcg(rb + t);
            a += x.x;
            z += x.y;
        }
        a = warp_sum(a);
        z = warp_sum(z);
        if (lane == 0) {
            S.r[Lr] = a;
            S.z[Lr] = z;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int j = 0;
        for (int Lc = 1; Lc <= ke; ++Lc) {
            const float w = __ldcg(&P.bpend[(int64_t)b * rpr + Lc].z);
            float h = w;
            if (Lc < ke) {
                const float denom = S.r[Lc] + 1.f - w;
                h = denom > 0.f ? S.r[Lc] / denom : 1.f;
            }
            if (uniforms(P, (uint32_t)(Lc - 1), (uint32_t)b).x < h) j = Lc;
        }
        const int use_p = (j == ke) || !(S.r[j] > 0.f);
        S.j = j;
        S.use_p = use_p;
        S.Z = use_p ? S.z[j] : S.r[j];
        S.t = uniforms(P, (uint32_t)j, (uint32_t)b).y * S.Z;
    }
    __syncthreads();
    const int j = S.j;
    const float2 *rb = P.recs3 + ((int64_t)b * rpr + j) * per_row;
    ResidSmem &F = S.R;
    if (warp == 0) {
        float cum = 0.f, before = 0.f, lp_before = 0.f;
        int found = -1, lastpos = -1;
        const float t = S.t;
        for (int c0 = 0; c0 < per_row; c0 += 32) {
            const int ti = c0 + lane;
            float m = 0.f;
            if (ti < per_row) {
                const float2 x = __ldcg(rb + ti);
                m = S.use_p ? x.y : x.x;
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
        }
    }
    __syncthreads();
    int drawn = -1;
    if (F.rec >= 0) {
        const int rc = F.rec / NW, rw = F.rec % NW;
        const int64_t a0 = (int64_t)rc * P.Ec2, a1 = min(a0 + P.Ec2, V);
        const int64_t sp = (a1 - a0 + NW - 1) / NW;
        const int64_t s0 = min(a0 + rw * sp, a1), s1 = SV_INB(min(s0 + sp, a1) - 1, V, 607) ? min(s0 + sp, a1) : s0;
        const float4 bp = P.bpend[(int64_t)b * rpr + j];
        const int64_t r = (int64_t)b * rpr + j;
        const void *row = reinterpret_cast<const T *>(P.logits) + r * V;
        const float *qrow = (j < P.k && !S.use_p) ? P.q + ((int64_t)b * P.k + j) * V : nullptr;
        ResidSrc<T> src{row, qrow, s0, s1, P.cs, bp.x, 1.f / bp.y, S.use_p, bp.z, NEG_INF};
        draw_init(F.D, F.cum_before);
        draw_span<2>(src, (s1 - s0 + 7) / 8, F.take_last ? POS_INF : S.t, F.D);
        drawn = F.D.found >= 0 ? F.D.found : F.D.lastpos;
    }
    int32_t *ot = P.out_tokens + (int64_t)b * (P.k + 1);
    for (int i = tid; i <= P.k; i += NT) {
        int v = -1;
        if (i < j && SV_INB((int64_t)b * P.k + i, (int64_t)P.B * P.k, 608)) v = __ldg(P.drafts + (int64_t)b * P.k + i);
        else if (i == j) v = drawn >= 0 ? drawn : 0;
        if (SV_INB((int64_t)b * (P.k + 1) + i, (int64_t)P.B * (P.k + 1), 609)) ot[i] = v;
    }
    if (tid == 0) {
        P.accept_len[b] = j;
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

// Column chunks per request of the residual and block kernels: about SV_RESID_TARGET CTAs in all,
// and at least four per request, so that at large B a request's re-read is spread over more SMs
// (B = 512, one draft: 109.8 to 100.3 us per call with four instead of two).
static int residual_chunks(int B, int64_t V)
{
    int64_t want = (SV_RESID_TARGET + B - 1) / B;
    if (want < 4) want = 4;
    const int64_t cap = (V + 1023) / 1024;
    int64_t c = want < cap ? want : cap;
    if (c < 1) c = 1;
    if (c > C2_MAX) c = C2_MAX;
    return (int)c;
}

struct Layout {
    size_t cnt2, recs, caps, thr, pend, recs2, bpend, recs3, total;
};


// Streaming chunks per row for elements of `vec` per 16-byte vector (see chunk_of).
static int64_t chunks_per_row(int64_t V, int vec)
{
    const int64_t ce = (int64_t)CHUNK_VEC * vec;
    return (V + vec - 1 + ce - 1) / ce;
}

// Streaming CTAs (one per SM at most) and the chunks each takes.
static void plan_chunks(int64_t nchunks, int sms, int &G, int64_t &cpc)
{
    int64_t g = sms < 1 ? 1 : sms;
    if (g > nchunks) g = nchunks;
    cpc = (nchunks + g - 1) / g;
    G = (int)((nchunks + cpc - 1) / cpc);
}

static Layout layout(int B, int rpr, int64_t V, bool block = false)
{
    // The arrival counters sit in a fixed region at the start of every layout, so a workspace
    // shared by calls of different shapes never finds another call's records where its counters
    // are: every call leaves that region zero, whatever the shape of the next call.
    const int64_t R = (int64_t)B * rpr;
    const int C2 = residual_chunks(B, V);
    const int64_t nch = chunks_per_row(V, 4);  // fp32 logits need the most chunks
    Layout L;
    size_t off = 0;
    L.cnt2 = off;
    off += sizeof(unsigned) * (size_t)B_MAX;
    L.recs = off;
    off += align256(sizeof(float4) * (size_t)R * nch);
    L.caps = off;
    off += align256(sizeof(float) * (size_t)R);
    L.thr = off;
    off += align256(sizeof(float) * (size_t)R);
    L.pend = off;
    off += align256(sizeof(int4) * (size_t)B);
    L.recs2 = off;
    off += align256(sizeof(float2) * (size_t)B * C2 * NW);
    L.bpend = off;
    L.recs3 = off;
    if (block) {
        off += align256(sizeof(float4) * (size_t)R);
        L.recs3 = off;
        off += align256(sizeof(float2) * (size_t)R * C2 * NW);
    }
    L.total = off;
    return L;
}

struct DevInfo {
    int sms = 0;
    int smem_sm = 0;        // shared memory per SM
    int fin_smem_max = 0;   // dynamic shared memory the finalising kernels may request
    int fin_static = 0;     // their static shared memory as the runtime counts it
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
        cudaGetLastError();
        d.sms = sms;
    }
    if (d.fin_smem_max == 0) {
        // The finalising kernels take dynamic shared memory only to limit how many of their CTAs
        // share an SM (see fin_dyn_smem); they are allowed up to the per-CTA maximum once per
        // device.  That maximum is the opt-in limit less the kernel's static shared memory as the
        // runtime counts it (FinSmem, padded to the alignment of the module's dynamic part).
        int smem_sm = 0, optin = 0;
        if (cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        const void *fins[] = {(const void *)sv_finalize_kernel<__nv_bfloat16, false, false>,
                              (const void *)sv_finalize_kernel<__nv_bfloat16, true, false>,
                              (const void *)sv_finalize_kernel<__nv_bfloat16, true, true>,
                              (const void *)sv_finalize_kernel<float, false, false>,
                              (const void *)sv_finalize_kernel<float, true, false>,
                              (const void *)sv_finalize_kernel<float, true, true>};
        size_t st = 0;
        for (const void *f : fins) {
            cudaFuncAttributes fa;
            if (cudaFuncGetAttributes(&fa, f) != cudaSuccess) {
                cudaGetLastError();
                return nullptr;
            }
            if (fa.sharedSizeBytes > st) st = fa.sharedSizeBytes;
        }
        const int mx = optin - (int)st;
        const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
        bool ok = mx > 0 && cudaFuncSetAttribute((const void *)sv_topkp_ring_kernel<__nv_bfloat16>, attr,
                                                 (int)sizeof(RingSmem)) == cudaSuccess;
        for (const void *f : fins) ok = ok && cudaFuncSetAttribute(f, attr, mx) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            return nullptr;
        }
        d.smem_sm = smem_sm;
        d.fin_static = (int)st;
        d.fin_smem_max = mx;
    }
    return &d;
}


static int common_setup(Params &P, const void *logits, int dtype, int B, int rpr, int64_t V,
                        void *workspace, size_t ws_bytes, bool block = false)
{
    if (!logits || !workspace) return SPEC_VERIFY_EINVAL;
    if (dtype != SPEC_VERIFY_BF16 && dtype != SPEC_VERIFY_FP32) return SPEC_VERIFY_EINVAL;
    const int esize = dtype == SPEC_VERIFY_BF16 ? 2 : 4;
    if ((uintptr_t)logits % esize) return SPEC_VERIFY_EINVAL;
    if ((uintptr_t)workspace % 256) return SPEC_VERIFY_EWORKSPACE;
    const Layout L = layout(B, rpr, V, block);
    if (ws_bytes < L.total) return SPEC_VERIFY_EWORKSPACE;
    const DevInfo *d = device_info();
    if (!d) return SPEC_VERIFY_ECUDA;
    char *ws = static_cast<char *>(workspace);
    P.logits = logits;
    P.thr_single = 1.f;
    P.thr_acc = 1.f;
    P.B = B;
    P.rpr = rpr;
    P.V = V;
    P.total = (int64_t)B * rpr * V;
    P.nch = chunks_per_row(V, esize == 2 ? 8 : 4);
    P.nchunks = (int64_t)B * rpr * P.nch;
    plan_chunks(P.nchunks, d->sms, P.G, P.cpc);
    P.mis = (int)(((uintptr_t)logits % 16) / esize);
    P.cnt2 = reinterpret_cast<unsigned *>(ws + L.cnt2);
    P.recs = reinterpret_cast<float4 *>(ws + L.recs);
    P.caps = reinterpret_cast<float *>(ws + L.caps);
    P.thr = reinterpret_cast<float *>(ws + L.thr);
    P.pend = reinterpret_cast<int4 *>(ws + L.pend);
    P.recs2 = reinterpret_cast<float2 *>(ws + L.recs2);
    P.bpend = reinterpret_cast<float4 *>(ws + L.bpend);
    P.recs3 = reinterpret_cast<float2 *>(ws + L.recs3);
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

// Dynamic shared memory for the finalising kernel's launch.  Its CTAs are placed as the streaming
// CTAs leave their SMs, and without a limit the first SMs to empty take as many as fit (eight),
// which then share one SM's issue slots and special-function units while most SMs idle.  Asking
// for a share of the SM's shared memory caps them at ceil(B / SMs) per SM: one per SM whenever
// the batch has no more requests than the GPU has SMs.
static size_t fin_dyn_smem(const DevInfo &d, int B)
{
    int per_sm = (B + d.sms - 1) / d.sms;
    if (per_sm > 2048 / NT_FIN_MAX) return 0;  // as many as the SM's threads allow anyway
    const int reserve = 1024;                  // shared memory the system keeps per CTA
    int dyn = d.smem_sm / per_sm - d.fin_static - reserve;
    if (dyn > d.fin_smem_max) dyn = d.fin_smem_max;
    return dyn > 0 ? (size_t)dyn : 0;
}

template <bool SAMPLE>
static int launch_stream(const Params &P, int dtype, cudaStream_t s)
{
    const DevInfo *dinfo = device_info();
    if (!dinfo) return SPEC_VERIFY_ECUDA;
    // The finaliser is launched as a programmatic dependent of the streaming kernel: its CTAs may
    // start early, stage the request's inputs, and wait (griddepcontrol) for the records.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P.B);
    cfg.blockDim = dim3(NT_FIN_MAX);  // one warp per row (rows beyond 8 loop); the rescan wants all 8
    cfg.dynamicSmemBytes = fin_dyn_smem(*dinfo, P.B);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool filt = SAMPLE && (P.top_k || P.top_p);
    const bool var = filt || P.temps || P.thr_single != 1.f || P.thr_acc != 1.f;
    if (filt) {  // each row's top-k / top-p threshold, before the rows are streamed
        // Rows in flight: TK_CTAS CTAs per SM, one row each (two per SM hold 304 rows, 78 MB of
        // bf16 rows of 128256, which L2 keeps for the row's later passes).
        const int64_t rows = (int64_t)P.B * P.rpr;
        const int64_t cap = TK_CTAS * (int64_t)dinfo->sms;
        const unsigned grid = (unsigned)(rows < cap ? rows : cap);
        if (dtype == SPEC_VERIFY_BF16) {
            // The ring kernel first (RING_CTAS CTAs per SM, one read of each row); the general one
            // takes the rows it leaves, launched as a programmatic dependent so that its launch
            // overlaps the ring kernel's last rows (it waits for the ring grid before reading).
            const int64_t ring_cap = (int64_t)RING_CTAS * dinfo->sms;
            const unsigned ring_grid = (unsigned)(rows < ring_cap ? rows : ring_cap);
            sv_topkp_ring_kernel<__nv_bfloat16><<<ring_grid, NT_RING + 32, sizeof(RingSmem), s>>>(P);
#if SV_PDL_TOPKP
            cudaLaunchConfig_t gcfg = {};
            gcfg.gridDim = dim3(grid);
            gcfg.blockDim = dim3(NT_TK);
            gcfg.stream = s;
            gcfg.attrs = attr;
            gcfg.numAttrs = 1;
            if (cudaLaunchKernelEx(&gcfg, sv_topkp_kernel<__nv_bfloat16>, P, 1) != cudaSuccess)
                return SPEC_VERIFY_ECUDA;
#else
            sv_topkp_kernel<__nv_bfloat16><<<grid, NT_TK, 0, s>>>(P, 1);
#endif
        } else {
            sv_topkp_kernel<float><<<grid, NT_TK, 0, s>>>(P, 0);
        }
        if (cudaGetLastError() != cudaSuccess) return SPEC_VERIFY_ECUDA;
    }
    if (dtype == SPEC_VERIFY_BF16) {
        if (filt && !P.temps) sv_stream_kernel<__nv_bfloat16, 4><<<P.G, stream_threads(4), 0, s>>>(P);
        else if (filt) sv_stream_kernel<__nv_bfloat16, 3><<<P.G, stream_threads(3), 0, s>>>(P);
        else if (P.temps) sv_stream_kernel<__nv_bfloat16, 2><<<P.G, stream_threads(2), 0, s>>>(P);
        else sv_stream_kernel<__nv_bfloat16, SAMPLE ? 1 : 0><<<P.G, NT_S, 0, s>>>(P);
        if (cudaGetLastError() != cudaSuccess) return SPEC_VERIFY_ECUDA;
        if (cudaLaunchKernelEx(&cfg, SAMPLE && var ? sv_finalize_kernel<__nv_bfloat16, SAMPLE, true>
                                                   : sv_finalize_kernel<__nv_bfloat16, SAMPLE, false>,
                               P) != cudaSuccess)
            return SPEC_VERIFY_ECUDA;
    } else {
        if (filt && !P.temps) sv_stream_kernel<float, 4><<<P.G, stream_threads(4), 0, s>>>(P);
        else if (filt) sv_stream_kernel<float, 3><<<P.G, stream_threads(3), 0, s>>>(P);
        else if (P.temps) sv_stream_kernel<float, 2><<<P.G, stream_threads(2), 0, s>>>(P);
        else sv_stream_kernel<float, SAMPLE ? 1 : 0><<<P.G, NT_S, 0, s>>>(P);
        if (cudaGetLastError() != cudaSuccess) return SPEC_VERIFY_ECUDA;
        if (cudaLaunchKernelEx(&cfg, SAMPLE && var ? sv_finalize_kernel<float, SAMPLE, true>
                                               : sv_finalize_kernel<float, SAMPLE, false>,
                               P) != cudaSuccess)
            return SPEC_VERIFY_ECUDA;
    }
    return cudaGetLastError() == cudaSuccess ? SPEC_VERIFY_OK : SPEC_VERIFY_ECUDA;
}

static bool temperature_ok(float t) { return t > 0.f && std::isfinite(t); }

// The argument checks of spec_verify_rejection that need no workspace.
static bool rejection_args_ok(const void *logits, int dtype, const int32_t *draft_ids, const float *draft_probs,
                              int B, int k, int V, float temperature, const int32_t *out_tokens,
                              const int32_t *accept_len)
{
    if (B < 1 || B > B_MAX || k < 0 || k + 1 > MAX_RPR || V < 1) return false;
    if ((k > 0 && !draft_ids) || !out_tokens || !accept_len) return false;
    if (!temperature_ok(temperature)) return false;
    if (draft_probs && ((uintptr_t)draft_probs % 4)) return false;
    if (!logits || (dtype != SPEC_VERIFY_BF16 && dtype != SPEC_VERIFY_FP32)) return false;
    if ((uintptr_t)logits % (dtype == SPEC_VERIFY_BF16 ? 2 : 4)) return false;
    const int64_t nch = chunks_per_row(V, dtype == SPEC_VERIFY_BF16 ? 8 : 4);
    return (int64_t)B * (k + 1) * nch < ((int64_t)1 << 31);
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_verify_workspace_bytes(int mode, int B, int k_or_N, int V)
{
    if (B < 1 || B > B_MAX || V < 1) return 0;
    int rpr;
    if (mode == SPEC_VERIFY_MODE_GREEDY || mode == SPEC_VERIFY_MODE_REJECTION || mode == SPEC_VERIFY_MODE_BLOCK) {
        if (k_or_N < 0 || k_or_N + 1 > MAX_RPR) return 0;
        rpr = k_or_N + 1;
    } else if (mode == SPEC_VERIFY_MODE_TREE) {
        if (k_or_N < 1 || k_or_N > MAX_RPR) return 0;
        rpr = k_or_N;
    } else {
        return 0;
    }
    return layout(B, rpr, V, mode == SPEC_VERIFY_MODE_BLOCK).total;
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
    case SPEC_VERIFY_DEV_BAD_KV_POSITION: return "device: KV compaction positions outside the slot table";
    case SPEC_VERIFY_DEV_BAD_KV_SLOT: return "device: KV compaction slot outside the pool";
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
    int rc = common_setup(P, logits, dtype, B, k + 1, V, workspace, ws_bytes);
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
    if (!rejection_args_ok(logits, dtype, draft_ids, draft_probs, B, k, V, temperature, out_tokens, accept_len))
        return SPEC_VERIFY_EINVAL;
    Params P;
    memset(&P, 0, sizeof P);
    int rc = common_setup(P, logits, dtype, B, k + 1, V, workspace, ws_bytes);
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

int spec_verify_block(const void *logits, int dtype, const int32_t *draft_ids, const float *draft_probs,
                      int B, int k, int V, float temperature, uint64_t seed, uint64_t offset,
                      int32_t *out_tokens, int32_t *accept_len, void *workspace, size_t ws_bytes,
                      int32_t *dev_status, void *stream)
{
    if (B < 1 || B > B_MAX || k < 0 || k + 1 > MAX_RPR || V < 1) return SPEC_VERIFY_EINVAL;
    if ((k > 0 && !draft_ids) || !out_tokens || !accept_len) return SPEC_VERIFY_EINVAL;
    if (!temperature_ok(temperature)) return SPEC_VERIFY_EINVAL;
    if (draft_probs && ((uintptr_t)draft_probs % 4)) return SPEC_VERIFY_EINVAL;
    Params P;
    memset(&P, 0, sizeof P);
    int rc = common_setup(P, logits, dtype, B, k + 1, V, workspace, ws_bytes, true);
    if (rc) return rc;
    P.drafts = draft_ids;
    P.q = (k > 0) ? draft_probs : nullptr;
    P.k = k;
    P.is_tree = 0;
    P.block = 1;
    P.out_tokens = out_tokens;
    P.accept_len = accept_len;
    P.dev_status = dev_status;
    set_rng(P, temperature, seed, offset);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = launch_stream<true>(P, dtype, s);
    if (rc || !P.q) return rc;
    const unsigned grid = (unsigned)P.C2 * (unsigned)(k + 1) * (unsigned)B;
    if (dtype == SPEC_VERIFY_BF16)
        sv_block_kernel<__nv_bfloat16><<<grid, NT, 0, s>>>(P);
    else
        sv_block_kernel<float><<<grid, NT, 0, s>>>(P);
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
    int rc = common_setup(P, logits, dtype, B, N, V, workspace, ws_bytes);
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

static bool thresholds_ok(const spec_verify_options *opt)
{
    return opt->threshold_single > 0.f && opt->threshold_single <= 1.f && opt->threshold_acc > 0.f &&
           opt->threshold_acc <= 1.f;
}

int spec_verify_rejection_ex(const void *logits, int dtype, const int32_t *draft_ids,
                             const float *draft_probs, int B, int k, int V,
                             const spec_verify_options *opt, uint64_t seed, uint64_t offset,
                             int32_t *out_tokens, int32_t *accept_len, float *out_probs,
                             void *workspace, size_t ws_bytes, int32_t *dev_status, void *stream)
{
    if (!opt || !thresholds_ok(opt)) return SPEC_VERIFY_EINVAL;
    if (draft_probs && (opt->threshold_single != 1.f || opt->threshold_acc != 1.f)) return SPEC_VERIFY_EINVAL;
    if ((uintptr_t)opt->temperatures % 4 || (uintptr_t)opt->top_k % 4 || (uintptr_t)opt->top_p % 4)
        return SPEC_VERIFY_EINVAL;
    const float T = opt->temperature;
    if (!opt->temperatures && !(T == 0.f || temperature_ok(T))) return SPEC_VERIFY_EINVAL;
    if (!opt->temperatures && T == 0.f) {  // an all-greedy batch; out_probs, if given, are 0
        int rc = spec_verify_greedy(logits, dtype, draft_ids, B, k, V, out_tokens, accept_len, workspace,
                                    ws_bytes, dev_status, stream);
        if (rc == SPEC_VERIFY_OK && out_probs &&
            cudaMemsetAsync(out_probs, 0, sizeof(float) * 3 * (size_t)B * (size_t)(k + 1),
                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
            rc = SPEC_VERIFY_ECUDA;
        return rc;
    }
    if (B < 1 || B > B_MAX || k < 0 || k + 1 > MAX_RPR || V < 1) return SPEC_VERIFY_EINVAL;
    if ((k > 0 && !draft_ids) || !out_tokens || !accept_len) return SPEC_VERIFY_EINVAL;
    if (draft_probs && ((uintptr_t)draft_probs % 4)) return SPEC_VERIFY_EINVAL;
    Params P;
    memset(&P, 0, sizeof P);
    int rc = common_setup(P, logits, dtype, B, k + 1, V, workspace, ws_bytes);
    if (rc) return rc;
    P.drafts = draft_ids;
    P.q = (k > 0) ? draft_probs : nullptr;
    P.k = k;
    P.is_tree = 0;
    P.out_tokens = out_tokens;
    P.accept_len = accept_len;
    P.out_probs = out_probs;
    P.dev_status = dev_status;
    set_rng(P, opt->temperatures ? 1.f : T, seed, offset);
    P.temps = opt->temperatures;
    P.thr_single = opt->threshold_single;
    P.thr_acc = opt->threshold_acc;
    P.top_k = opt->top_k;
    P.top_p = opt->top_p;
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

int spec_verify_tree_ex(const void *logits, int dtype, const int32_t *node_tokens,
                        const int32_t *parents, int B, int N, int V, const spec_verify_options *opt,
                        uint64_t seed, uint64_t offset, int32_t *out_tokens, int32_t *accept_index,
                        int32_t *accept_len, void *workspace, size_t ws_bytes, int32_t *dev_status,
                        void *stream)
{
    if (!opt || !thresholds_ok(opt)) return SPEC_VERIFY_EINVAL;
    if ((uintptr_t)opt->temperatures % 4 || (uintptr_t)opt->top_k % 4 || (uintptr_t)opt->top_p % 4)
        return SPEC_VERIFY_EINVAL;
    const float T = opt->temperature;
    if (!opt->temperatures && !(T == 0.f || temperature_ok(T))) return SPEC_VERIFY_EINVAL;
    if (B < 1 || B > B_MAX || N < 1 || N > MAX_RPR || V < 1) return SPEC_VERIFY_EINVAL;
    if (!node_tokens || !parents || !out_tokens || !accept_index || !accept_len) return SPEC_VERIFY_EINVAL;
    Params P;
    memset(&P, 0, sizeof P);
    int rc = common_setup(P, logits, dtype, B, N, V, workspace, ws_bytes);
    if (rc) return rc;
    P.node_tokens = node_tokens;
    P.parents = parents;
    P.k = N - 1;
    P.is_tree = 1;
    P.out_tokens = out_tokens;
    P.accept_index = accept_index;
    P.accept_len = accept_len;
    P.dev_status = dev_status;
    P.thr_single = opt->threshold_single;
    P.thr_acc = opt->threshold_acc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!opt->temperatures && T == 0.f) return launch_stream<false>(P, dtype, s);
    set_rng(P, opt->temperatures ? 1.f : T, seed, offset);
    P.temps = opt->temperatures;
    P.top_k = opt->top_k;
    P.top_p = opt->top_p;
    return launch_stream<true>(P, dtype, s);
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

namespace sv {
unsigned long long kv_debug_fault();
unsigned long long budget_debug_fault();
}  // namespace sv

// The first out-of-range index the kernels met (debug builds), read and cleared across the
// library's three modules; synchronous (symbol copies).
extern "C" int spec_verify_debug_fault(uint64_t *fault)
{
    if (!fault) return SPEC_VERIFY_EINVAL;
    unsigned long long w = 0;
#ifdef SV_DEBUG
    unsigned long long z = 0;
    if (cudaMemcpyFromSymbol(&w, sv::g_sv_debug_fault, sizeof w) != cudaSuccess ||
        cudaMemcpyToSymbol(sv::g_sv_debug_fault, &z, sizeof z) != cudaSuccess)
        return SPEC_VERIFY_ECUDA;
#endif
    const unsigned long long kv = sv::kv_debug_fault(), bu = sv::budget_debug_fault();
    if (kv == ~0ull || bu == ~0ull) return SPEC_VERIFY_ECUDA;
    *fault = w ? w : (kv ? kv : bu);
    return SPEC_VERIFY_OK;
}

// Stage waits of the threshold ring kernel that ran out of time, read and cleared; synchronous.
extern "C" int spec_verify_wait_timeouts(uint64_t *count)
{
    if (!count) return SPEC_VERIFY_EINVAL;
    unsigned long long n = 0, z = 0;
    if (cudaMemcpyFromSymbol(&n, sv::g_ring_timeouts, sizeof n) != cudaSuccess ||
        cudaMemcpyToSymbol(sv::g_ring_timeouts, &z, sizeof z) != cudaSuccess)
        return SPEC_VERIFY_ECUDA;
    *count = n;
    return SPEC_VERIFY_OK;
}

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
    // Every argument check comes first, so that a rejected call enqueues nothing.
    if (!rejection_args_ok(logits, dtype, draft_ids, draft_probs, B, k, V, temperature, out_tokens, accept_len))
        return SPEC_VERIFY_EINVAL;
    const size_t need = spec_verify_workspace_bytes(SPEC_VERIFY_MODE_REJECTION, B, k, V);
    if (need == 0) return SPEC_VERIFY_EINVAL;
    if (need > SPEC_VERIFY_NOALLOC_SCRATCH_BYTES) return SPEC_VERIFY_ETOOBIG;
    if (!device_info()) return SPEC_VERIFY_ECUDA;
    void *scratch = noalloc_scratch_address();
    if (!scratch) return SPEC_VERIFY_ECUDA;
    // The scratch keeps whatever the previous call left; the arrival counters of the requests
    // this call uses must start at zero (every completed call leaves them zero, but a call cut
    // short may not), so clear them (a memset, no allocation).
    const Layout L = layout(B, k + 1, V);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(scratch);
    if (cudaMemsetAsync(base + L.cnt2, 0, sizeof(unsigned) * (size_t)B, s) != cudaSuccess)
        return SPEC_VERIFY_ECUDA;
    return spec_verify_rejection(logits, dtype, draft_ids, draft_probs, B, k, V, temperature, seed,
                                 offset, out_tokens, accept_len, out_probs, scratch,
                                 SPEC_VERIFY_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
