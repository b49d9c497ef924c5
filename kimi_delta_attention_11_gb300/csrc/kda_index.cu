// kda_index.cu -- chunk index of fixed-length or packed variable-length input.
//
// Tokamax "chunk_kda_fwd_design_doc", 3.5 (single-alignment contract) and 9.1.7
// (variable-length sequences): sequence n covers tokens [p_n, p_{n+1}); it is cut into
// chunks of C tokens, the last one shorter when L_n is not a multiple of C, so a chunk
// never crosses two sequences.  The design doc pads every segment to C * ceil(L_n / C)
// physically; here the padding exists only in the index (a chunk carries its length)
// and the kernels mask the missing rows, so no padded copy of the input is made.
//
// One CTA of 1024 threads: a block-wide exclusive scan of per-sequence chunk counts
// (tiles of 1024 sequences), then every thread fills chunk entries by a binary search
// over the sequence table.  Everything stays on the device: the host never waits for
// the chunk count, the consumer kernels are launched over an upper bound and their
// surplus CTAs exit.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kThreads = 1024;

__device__ __forceinline__ void seq_bounds(const int32_t* cu, int n, int T, int* start, int* len) {
    if (cu) {
        const int a = cu[n], b = cu[n + 1];
        *start = a;
        *len = b > a ? b - a : 0;  // a decreasing offset pair is an empty sequence
    } else {
        *start = n * T;
        *len = T;
    }
}

__global__ void __launch_bounds__(kThreads)
chunk_index_kernel(const int32_t* __restrict__ cu, int N, int T, int4* __restrict__ chunk_tab,
                   int2* __restrict__ seq_tab, int* __restrict__ count, long long max_chunks) {
    __shared__ int warp_tot[kThreads / 32];
    __shared__ int s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_carry = 0;
    __syncthreads();

    // Phase 1: seq_tab[n] = {first chunk, chunk count}, exclusive scan over n.
    for (int base = 0; base < N; base += kThreads) {
        const int n = base + tid;
        int start = 0, len = 0;
        if (n < N) seq_bounds(cu, n, T, &start, &len);
        const int cnt = (len + kChunk - 1) / kChunk;
        int incl = cnt;  // warp inclusive scan
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = warp_tot[lane];
            int wi = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, wi, off);
                if (lane >= off) wi += y;
            }
            warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
        }
        __syncthreads();
        const int first = s_carry + warp_tot[warp] + incl - cnt;
        if (n < N) seq_tab[n] = make_int2(first, cnt);
        __syncthreads();
        if (tid == kThreads - 1) s_carry = first + cnt;
        __syncthreads();
    }
    const int total = s_carry;
    if (tid == 0) *count = total;

    // Phase 2: chunk_tab[c] for every chunk; the sequence of c is the last n whose
    // first chunk is <= c.
    for (long long c = tid; c < total && c < max_chunks; c += kThreads) {
        int lo = 0, hi = N - 1;
        while (lo < hi) {  // last n with seq_tab[n].x <= c
            const int mid = (lo + hi + 1) >> 1;
            if (seq_tab[mid].x <= c) lo = mid; else hi = mid - 1;
        }
        // an empty sequence shares its first index with the next non-empty one, which
        // the search prefers, so seq_tab[lo] always has at least one chunk here
        const int n = lo;
        int start, len;
        seq_bounds(cu, n, T, &start, &len);
        const int j = (int)c - seq_tab[n].x;
        const int clen = min(kChunk, len - j * kChunk);
        chunk_tab[c] = make_int4(n, start + j * kChunk, clen, j);
    }
}

}  // namespace

cudaError_t launch_chunk_index(const int32_t* cu_seqlens, int N, int T, const Layout& L,
                               char* ws, cudaStream_t s) {
    chunk_index_kernel<<<1, kThreads, 0, s>>>(
        cu_seqlens, N, T, reinterpret_cast<int4*>(ws + L.chunk_tab_off),
        reinterpret_cast<int2*>(ws + L.seq_tab_off), reinterpret_cast<int*>(ws + L.count_off),
        L.max_chunks);
    return cudaGetLastError();
}

}  // namespace kda
