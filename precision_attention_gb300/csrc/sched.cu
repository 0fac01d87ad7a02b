// sched.cu -- GPU-resident work list for the forward (no host synchronisation).
//
// FLAMIA: document-local scaling of packed documents without repacking
// (abstract, section 4.1); longest-first ordering of causal work (section 4.3:
// dropping it costs 10-65% of causal forward time); scales and work lists kept
// on the GPU so the call can be captured in a CUDA graph (appendix F).
#include <cuda_runtime.h>

#include "params.h"
#include "pdl.cuh"

namespace pa {

// exclusive scan of up to 4 * blockDim values held 4 per thread; returns the total
__device__ int block_exclusive_scan4(int (&v)[4], int* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int acc = v[0] + v[1] + v[2] + v[3];
    int inc = acc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += x;
    }
    __syncthreads();
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    int base = 0, total = 0;
    for (int w = 0; w < nw; w++) {
        if (w < warp) base += wsum[w];
        total += wsum[w];
    }
    int run = base + inc - acc;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const int c = v[k];
        v[k] = run;
        run += c;
    }
    return total;
}

__global__ void __launch_bounds__(1024) sched_kernel(SchedParams p) {
    __shared__ int wsum[32];
    __shared__ int bad;
    // reads only cu_seqlens and writes only the work list and the header's counts,
    // which the quantiser before it neither reads nor writes: it runs beside the
    // quantiser's last tiles; the V-reference pass may be scheduled meanwhile
    pdl_trigger();
    const int tid = threadIdx.x, nd = p.nd;
    if (tid == 0) bad = 0;
    __syncthreads();
    // pass 1: document table (4 documents per thread per round)
    int carry_t = 0, carry_q = 0, carry_k = 0, carry_v = 0, carry_p = 0;
    for (int base = 0; base < nd; base += 4 * blockDim.x) {
        int nt[4], nq[4], nk[4], nv[4], np[4], st[4], ln[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int i = base + tid * 4 + k;
            nt[k] = nq[k] = nk[k] = nv[k] = np[k] = st[k] = ln[k] = 0;
            if (i < nd) {
                const int s = p.cu ? p.cu[i] : 0, e = p.cu ? p.cu[i + 1] : p.T;
                if (e < s) bad = 1;
                const int L = e > s ? e - s : 0;
                st[k] = s;
                ln[k] = L;
                nt[k] = (L + 127) / 128;
                np[k] = (nt[k] + 1) / 2;
                nq[k] = (L + p.bq - 1) / p.bq;
                nk[k] = (L + p.bk - 1) / p.bk;
                nv[k] = (L + p.bv - 1) / p.bv;
            }
        }
        const int tt = block_exclusive_scan4(nt, wsum);
        const int tq = block_exclusive_scan4(nq, wsum);
        const int tk = block_exclusive_scan4(nk, wsum);
        const int tv = block_exclusive_scan4(nv, wsum);
        const int tp = block_exclusive_scan4(np, wsum);
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int i = base + tid * 4 + k;
            if (i < nd) {
                DocEntry d;
                d.start = st[k];
                d.len = ln[k];
                d.toff = carry_t + nt[k];
                d.boff_q = carry_q + nq[k];
                d.boff_k = carry_k + nk[k];
                d.boff_v = carry_v + nv[k];
                d.poff = carry_p + np[k];
                d.pad1 = 0;
                p.docs[i] = d;
            }
        }
        carry_t += tt;
        carry_q += tq;
        carry_k += tk;
        carry_v += tv;
        carry_p += tp;
    }
    if (tid == 0) {
        const int c0 = p.cu ? p.cu[0] : 0, cn = p.cu ? p.cu[nd] : p.T;
        if (c0 != 0 || cn != p.T) bad = 1;
    }
    __syncthreads();
    const int units = p.qpair ? carry_p : carry_t;     // query tiles or query-tile pairs
    const long long total = (long long)units * p.H;
    if (bad || total > p.items_cap) {
        if (tid == 0) {
            atomicOr(&p.hdr->status, ST_BAD_SEQLENS);
            p.hdr->n_items = 0;
            p.hdr->n_tiles = 0;
        }
        pdl_wait();   // this kernel's completion implies the previous one's
        return;
    }
    // pass 2: work items
    if (!p.causal) {
        // document, head, query tile: consecutive CTAs share a head's K and V in L2
        for (long long i = tid; i < total; i += blockDim.x) {
            int lo = 0, hi = nd - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                const int off = p.qpair ? p.docs[mid].poff : p.docs[mid].toff;
                if ((long long)off * p.H <= i) lo = mid; else hi = mid - 1;
            }
            const DocEntry d = p.docs[lo];
            const int nt = (d.len + 127) / 128;
            const int nu = p.qpair ? (nt + 1) / 2 : nt;
            const long long rem = i - (long long)(p.qpair ? d.poff : d.toff) * p.H;
            WorkItem w;
            w.doc = lo;
            w.head = (int)(rem / nu);
            w.qtile = (int)(rem % nu);
            w.ntiles = nt;
            p.items[i] = w;
        }
    } else {
        // longest first: query tile qt of a causal document visits qt + 1 key
        // tiles (a pair p visits min(2p + 2, tiles)); order by the unit index
        // descending, then document, then head
        for (long long pr = tid; pr < units; pr += blockDim.x) {
            int lo = 0, hi = nd - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                const int off = p.qpair ? p.docs[mid].poff : p.docs[mid].toff;
                if (off <= pr) lo = mid; else hi = mid - 1;
            }
            const int doc = lo;
            const int qt = (int)(pr - (p.qpair ? p.docs[doc].poff : p.docs[doc].toff));
            long long before = 0;   // units of every document with a larger index
            int rank = 0;           // earlier documents that also have unit qt
            for (int j = 0; j < nd; j++) {
                const int ntj = (p.docs[j].len + 127) / 128;
                const int nuj = p.qpair ? (ntj + 1) / 2 : ntj;
                if (nuj > qt + 1) before += nuj - qt - 1;
                if (j < doc && nuj > qt) rank++;
            }
            const int ntd = (p.docs[doc].len + 127) / 128;
            const long long base = (before + rank) * p.H;
            for (int h = 0; h < p.H; h++) {
                WorkItem w;
                w.doc = doc;
                w.head = h;
                w.qtile = qt;
                w.ntiles = p.qpair ? (2 * qt + 2 < ntd ? 2 * qt + 2 : ntd) : qt + 1;
                p.items[base + h] = w;
            }
        }
    }
    if (tid == 0) {
        p.hdr->n_items = (int)total;
        p.hdr->n_tiles = units;
        p.hdr->ticket = p.ticket0;   // the forward's CTAs take items 0 .. grid - 1 first
    }
    pdl_wait();   // this kernel's completion implies the previous one's
}

// V reference scales (E4M3 layouts): the scale every row's V ratios r = s_v / ref
// are taken against. Default: the maximum over the document's V blocks
// (vref[h][doc]). Causal-exact (block 1): the running maximum of the token
// scales over positions <= t of the document (vref[h][t]), so a row never
// sees a later token's scale.
__global__ void __launch_bounds__(256) vref_kernel(VrefParams p) {
    __shared__ float wmax[8];
    __shared__ float carry;
    pdl_trigger();   // the attention kernel may set up; it waits for this one before its reads
    pdl_wait();      // the work list and (through it) the quantiser's scales
    // this call's schedule: the work-list pass wrote no items when its cu_seqlens
    // were malformed (the status word's bits may be older than this call)
    if (p.hdr->n_items <= 0) return;
    const int h = blockIdx.x % p.H, doc = blockIdx.x / p.H;
    const DocEntry d = p.docs[doc];
    const long long base = (long long)h * p.sv_cap + d.boff_v;
    // block i's V scale: fp32 (E4M3 layouts) or 2^X from the exponent byte (MX token layout)
    auto sv_at = [&](int i) -> float {
        if (p.sv_e8) {
            const uint32_t b = p.sv_e8[base + i];
            return b ? __uint_as_float(b << 23) : 0.0f;
        }
        return p.sv[base + i];
    };
    const int n = (d.len + p.bv - 1) / p.bv;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (!p.exact) {
        float m = 0.0f;
        for (int i = threadIdx.x; i < n; i += 256) m = fmaxf(m, sv_at(i));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) wmax[warp] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            float r = wmax[0];
            for (int w = 1; w < 8; w++) r = fmaxf(r, wmax[w]);
            p.vref[(long long)h * p.nd + doc] = r;
            carry = r;
        }
        if (!p.tiles) return;
        __syncthreads();
        // each key tile's score multiplier and V ratio (one scale per 128-token tile)
        const float ref = carry;
        const float inv_ref = ref > 0.0f ? __fdiv_rn(1.0f, ref) : 0.0f;   // rounded once per document
        const int nt = (d.len + 127) / 128;
        for (int j = threadIdx.x; j < nt; j += 256) {
            const float ks = p.sk[(long long)h * p.sk_cap + d.boff_k + (128 * j) / p.bk];
            const float sv = sv_at((128 * j) / p.bv);
            const float rj = (sv > 0.0f && ref > 0.0f) ? __fmul_rn(sv, inv_ref) : 1.0f;
            p.tsc[(long long)h * p.tsc_cap + d.toff + j] = make_float4(ks * p.C, __log2f(rj), __fdiv_rn(1.0f, rj), 0.0f);
        }
        return;
    }
    if (threadIdx.x == 0) carry = 0.0f;
    __syncthreads();
    for (int c0 = 0; c0 < n; c0 += 256) {
        const int i = c0 + threadIdx.x;
        float v = i < n ? sv_at(i) : 0.0f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float x = __shfl_up_sync(0xFFFFFFFFu, v, o);
            if (lane >= o) v = fmaxf(v, x);
        }
        if (lane == 31) wmax[warp] = v;
        __syncthreads();
        float pre = carry;
        for (int w = 0; w < warp; w++) pre = fmaxf(pre, wmax[w]);
        v = fmaxf(v, pre);
        if (i < n) p.vref[(long long)h * p.T + d.start + i] = v;
        __syncthreads();
        if (threadIdx.x == 255) carry = v;
        __syncthreads();
    }
}

cudaError_t launch_sched(const SchedParams& p, cudaStream_t st) {
    return launch_pdl(sched_kernel, dim3(1), dim3(1024), 0, st, p);
}

cudaError_t launch_vref(const VrefParams& p, cudaStream_t st) {
    return launch_pdl(vref_kernel, dim3((unsigned)(p.H * p.nd)), dim3(256), 0, st, p);
}

}  // namespace pa
