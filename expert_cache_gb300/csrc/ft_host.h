// The host share of a decode call: the mailbox through which the decode kernel hands
// its deferred routes to the host branch and the join kernel takes the host partial
// back.  Plain layout, shared by the CUDA and the host C++ sources.
//
// [EXPLAINER §8.3] the CPU branch sits inside the captured path: stable pinned
//   input / output buffers and task descriptors per batch size, a persistent worker
//   pool pinned to physical cores, dequantisation inside the SIMD GEMV;
// [BWRATIO "代码全链路" §2] the GPU share keeps its routes (others -1 or weight 0),
//   the host share gets the complement, and the two partials are summed.
//
// Mailbox (pinned, device-mapped; offsets from mailbox_layout):
//   header  uint32 task   decode kernel -> host: 1 = a host share is published
//           uint32 done   host -> join kernel: 1 = y holds the host partial
//           int32  layer, B, k, n_def   the published call (n_def: deferred routes;
//                                       written by every call, 0 = nothing to join)
//           uint32 published            calls published (diagnostic)
//   x       bf16 [B_max, H]   the call's activations
//   def     int32 [B_max, k_max]   flat id of each deferred route, else -1
//   w       fp32 [B_max, k_max]    the routes' gates
//   y       fp32 [B_max, H]   the host partial
#pragma once
#include <stddef.h>
#include <stdint.h>

namespace ft {

struct MailboxHeader {
    uint32_t task;
    uint32_t done;
    int32_t layer, B, k, n_def;
    uint32_t published;
    uint32_t reserved[9];
};
static_assert(sizeof(MailboxHeader) == 64, "mailbox header is 64 bytes");

struct MailboxLayout {
    size_t x, def, w, y, bytes;
};

#ifdef __CUDACC__
__host__ __device__
#endif
inline MailboxLayout mailbox_layout(int H, int k_max, int B_max) {
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    MailboxLayout m;
    m.x = 256;
    m.def = m.x + up((size_t)B_max * H * 2);
    m.w = m.def + up((size_t)B_max * k_max * 4);
    m.y = m.w + up((size_t)B_max * k_max * 4);
    m.bytes = m.y + up((size_t)B_max * H * 4);
    return m;
}

}  // namespace ft

struct ft_host_branch;

namespace ft {

// What the cache needs to know of a host branch (ft_host.cpp).
struct HostBranchInfo {
    int L, E, H, I, k_max, B_max, format;
    const void* pool;
    void* mailbox;
};
bool host_branch_info(const ft_host_branch* hb, HostBranchInfo* out);
// The host GEMV of one token (x = 1.0) through each of the n records `flats` (gate 1),
// with every worker; seconds of wall time, or < 0 on a bad list.
double host_branch_run_flats(ft_host_branch* hb, const int32_t* flats, int n);

}  // namespace ft
