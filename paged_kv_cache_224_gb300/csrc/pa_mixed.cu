// The one-launch continuous-batching step, host side: the split of the SMs
// between the prompt chunks and the decodes, the workspace, and the launch
// (kernel in pa_mixed.cuh).
#include "pa_prefill.cuh"

namespace pa {
namespace {
using namespace pf;

// Time model of one CTA per SM, to split the SMs between the halves: a prefill
// CTA finishes a 128-key tile of 256 rows in about 1.785 us with 8 query heads
// per kv head and about 2.5 us with 2 or 4 (measured: the split that model
// gives put 32/8- and 16/8-head steps at their best, 0.311 and 0.305 ms,
// where the 1.785 us figure left the chunk's CTAs the long pole); a decode
// CTA streams about 61 GB/s, and all of them together about 6.4 TB/s; once
// the prefill CTAs are done they join the decode, so too many prefill CTAs
// cost little and too few a lot.  The split minimises the step; the count of
// prefill CTAs is even (the CTAs pair up on the SM pairs of a TPC: with an
// odd count the one prefill CTA that shared its pair with a decode CTA ran
// about a third longer than the rest).
int mixed_prefill_ctas(long long prefill_tiles, double decode_bytes, int sms, int group) {
    const double tile_s = group == 8 ? 1.785e-6 : 2.5e-6;
    int best = 2;
    double best_t = 1e30;
    for (int n = 2; n < sms; n += 2) {
        const double tp = (double)prefill_tiles * tile_s / n;
        const double cap = 6.4e12;
        const double bw = std::min(cap, (sms - n) * 61e9);
        const double t = decode_bytes <= tp * bw ? std::max(tp, decode_bytes / bw)
                                                 : tp + (decode_bytes - tp * bw) / cap;
        if (t < best_t) {
            best_t = t;
            best = n;
        }
    }
    return best;
}

}  // namespace

bool mixed_supported(int head_dim, int block_size, int group) {
    // one query head per kv head decodes better on the CUDA cores (two launches)
    return head_dim == kD && (group == 2 || group == 4 || group == 8) &&
           (block_size == 16 || block_size == 32 || block_size == 64 || block_size == 128);
}

int launch_mixed(pa_dtype dt, int block_size, int group, const PrefillParams &pp_in, const DecodeParams &dp,
                 void *workspace, size_t workspace_bytes, double decode_bytes, cudaStream_t stream) {
    if (!mixed_supported(kD, block_size, group)) return PA_ERR_UNSUPPORTED;
    if ((long long)pp_in.num_blocks * pp_in.num_kv_heads * block_size >= (1LL << 31)) return PA_ERR_UNSUPPORTED;
    if (pp_in.num_seqs < 1 || pp_in.num_seqs > kPrefillMaxSeqs) return PA_ERR_INVALID_ARG;
    MixedParams mp{};
    mp.pp = pp_in;
    mp.dp = dp;
    long long units = 0;
    const int rc = prefill_schedule(mp.pp, group, &units);
    if (rc != PA_OK) return rc;
    const int sms = sm_count();
    if (units == 0 || sms < 2) return PA_ERR_UNSUPPORTED;
    const PrefillWs ws = prefill_ws(sms, units);
    if (!workspace || workspace_bytes < ws.total()) return PA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_ALIGNMENT;
    char *base = static_cast<char *>(workspace);
    mp.pp.split = 1;
    mp.pp.part_o = reinterpret_cast<float *>(base);
    mp.pp.part_ml = reinterpret_cast<float2 *>(base + ws.o_bytes);
    mp.pp.counters = reinterpret_cast<unsigned *>(base + ws.cnt_off());
    mp.decode_next = reinterpret_cast<unsigned *>(base + ws.queue_off());
    mp.prefill_ctas = (int)std::min<long long>(mixed_prefill_ctas(mp.pp.total_tiles, decode_bytes, sms, group), mp.pp.total_tiles);
    mp.decode_units = dp.num_seqs * dp.num_kv_heads;
    return dt == PA_BF16 ? launch_mixed_bf16(block_size, group, mp, (unsigned)sms, stream)
                         : launch_mixed_f16(block_size, group, mp, (unsigned)sms, stream);
}

}  // namespace pa
