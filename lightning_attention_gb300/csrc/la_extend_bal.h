// la_extend_bal.h -- the balanced extend's records and launcher, shared by la_extend_bal.cu and
// la_api.cu (not part of the ABI).
#pragma once

#include "la_internal.h"

namespace la {

// Balanced extend for one-wave batches of skewed lengths (la_extend_bal.cu): a one-block plan
// cuts the longest requests into segments (each segment's CTA first forms its start state from
// the request's earlier tokens) and writes one SegRec per segment, in the order the segments'
// (segment, head) items are dealt to a persistent grid of one CTA per SM.
struct alignas(16) SegHeader {
    int nrec;     // records written
    int target;   // the chosen target item cost (tenths of a chunk)
    int pad0, pad1;
};
struct alignas(16) SegRec {
    int b, y0, len, slot;             // request, first token of the segment, its length, pool slot
    int sp, tslot, nchunks, flags;    // tracked token relative to the segment (len + 1: none) and
                                      // its slot; chunks of the segment; kRec* flags
    int a, nseg, pad0, pad1;          // segment start in the request (prologue tokens, a multiple
                                      // of the chunk length); segments of the request
};
constexpr int kRecLast = 4;           // the request's last segment: writes the final state
constexpr int kMaxBalRequests = 256;  // the plan's request limit
constexpr int kMaxBalRecs = 256;      // the plan's segment limit
// Scratch of the balanced extend: the header, the records and one read counter per
// (request, head); 16-byte aligned.
size_t bal_scratch_bytes(int B, int H);
// Only for p.group == 1 without a sequence split, B <= kMaxBalRequests and B H <= ctas.
cudaError_t launch_extend_bal(const ExtendParams &p, void *scratch, int ctas, cudaStream_t stream);

}  // namespace la
