// sv_ngram.cu -- prompt-lookup (n-gram) drafting on the GPU.
//
// Method ("Medusa, EAGLE and self-speculation", lookup_draft; "7.6 Speculative Decoding:
// Draft Models, Medusa, EAGLE & Lookahead", Exercise 4 ngram_draft): the tail is a
// sequence's last n tokens; its most recent earlier occurrence is the largest start i <=
// len - n - 1 whose n tokens equal the tail; the drafts are the (up to k) tokens that
// followed it, padded with the last token when asked (Exercise 4).  The drafter's q is
// one-hot on each draft, so its drafts verify with the greedy entries or, sampling, as a
// draft row that is -inf everywhere but the draft token.
//
// One CTA per sequence.  The search runs from the end of the history backwards in chunks
// of kChunk starts; consecutive threads test consecutive starts (coalesced loads, the n
// tokens of a start mostly served by L1), and the first chunk holding a match ends the
// search -- on copy-heavy text the latest occurrence is usually near the end.
#include "sv_checks.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kNgThreads = 256;
constexpr int kNgWarps = kNgThreads / 32;
constexpr int kChunk = kNgThreads * 16;

}  // namespace

__global__ void __launch_bounds__(kNgThreads)
    ngram_draft_kernel(const int32_t *__restrict__ history, int64_t stride, const int32_t *__restrict__ lengths,
                       int n, int k, int pad, int32_t *__restrict__ drafts, int32_t *__restrict__ count) {
    __shared__ int s_tail[kMaxNgram];
    __shared__ int s_best[kNgWarps];
    griddep_launch_next();
    griddep_wait();  // the caller's kernels may still be writing the history
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t seq = blockIdx.x;
    const int32_t *h = history + seq * stride;
    const int64_t Lr = lengths[seq];
    const int L = int(Lr < 0 ? 0 : (Lr > stride ? stride : Lr));  // a length past the row is clamped to it
    if (tid < n && L >= n && SV_IN(tid, kMaxNgram) && SV_IN(L - n + tid, stride)) s_tail[tid] = h[L - n + tid];
    __syncthreads();
    int best = -1;
    for (int hi = L - n - 1; hi >= 0 && best < 0; hi -= kChunk) {  // uniform over the CTA
        const int lo = hi - kChunk + 1 > 0 ? hi - kChunk + 1 : 0;
        int local = -1;
        for (int i = hi - tid; i >= lo && local < 0; i -= kNgThreads) {  // descending: the first hit is the latest
            bool same = true;
            for (int t = 0; t < n && same && SV_IN(i + t, L); ++t) same = __ldg(h + i + t) == s_tail[t];
            if (same) local = i;
        }
        local = warp_reduce(local, [](int a, int b) { return max(a, b); });
        if (lane == 0) s_best[warp] = local;
        __syncthreads();
        int b = s_best[0];
        for (int w = 1; w < kNgWarps; ++w) b = max(b, s_best[w]);
        best = b;
        __syncthreads();
    }
    // the continuation (at most k tokens, inside the history), then the padding
    int32_t *out = drafts + seq * k;
    int avail = 0;
    if (best >= 0) avail = min(k, L - (best + n));
    const int c = pad && L >= 1 ? k : avail;
    for (int m = tid; m < k; m += kNgThreads)
        out[m] = m < avail ? (SV_IN(best + n + m, L) ? __ldg(h + best + n + m) : -1)
                           : (m < c ? (SV_IN(L - 1, stride) ? __ldg(h + L - 1) : -1) : -1);
    if (tid == 0) count[seq] = c;
}

cudaError_t launch_ngram_draft(const int32_t *history, int64_t stride, const int32_t *lengths, int B, int n, int k,
                               int pad, int32_t *drafts, int32_t *count, cudaStream_t s) {
    return launch_after(ngram_draft_kernel, unsigned(B), kNgThreads, 0, s, history, stride, lengths, n, k, pad, drafts,
                        count);
}

}  // namespace sv
