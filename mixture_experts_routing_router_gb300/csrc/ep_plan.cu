// ep_plan.cu -- the host-side plan of the expert-parallel count-first exchange.
//
// afdEP-comm count-first validation record (.change, .setup; the fault patches
// P3 "count puts" and P4 "FFN publishes prefix sums"): with the experts split
// over the ranks of a node, every rank first publishes its per-expert counts
// (E int32 per rank, E*G in all); from those counts alone each rank knows,
// before any payload row moves, the slot in the owner's expert-contiguous
// receive buffer where each of its rows lands, how many rows it sends to and
// receives from every peer, and whether some receive buffer would overflow.
// The payload then moves straight into place, and the combine goes back along
// the same segments.  This file holds that arithmetic; moving the rows is the
// caller's transport (NCCL or gloo point-to-point, or device copies).
#include "common.cuh"

namespace {

// First expert of rank g when E experts are split over G ranks in contiguous,
// balanced blocks.
inline int first_expert(long long g, int E, int G) { return (int)(g * E / G); }

}  // namespace

extern "C" moe_status moe_ep_plan(int32_t experts, int32_t world, int32_t rank, int32_t capacity,
                                  const int32_t* counts_all, int32_t* send_offsets, int32_t* recv_offsets,
                                  int32_t* recv_slot, int32_t* peer_send, int32_t* peer_recv) {
    using namespace moe;
    clear_error();
    const int E = experts, G = world;
    if (E < 1 || E > 1024 || G < 1 || G > E || rank < 0 || rank >= G || capacity < 1 || !counts_all ||
        !send_offsets || !recv_offsets || !recv_slot || !peer_send || !peer_recv) {
        set_error("moe_ep_plan: bad arguments (experts %d, world %d, rank %d, capacity %d)", E, G, rank, capacity);
        return MOE_ERR_INVALID_ARG;
    }
    for (long long i = 0; i < (long long)G * E; ++i)
        if (counts_all[i] < 0) {
            set_error("moe_ep_plan: negative count at [%lld, %lld]", i / E, i % E);
            return MOE_ERR_INVALID_ARG;
        }
    const int e0 = first_expert(rank, E, G), e1 = first_expert(rank + 1, E, G), el = e1 - e0;
    const int32_t* mine = counts_all + (size_t)rank * E;

    // sender side: this rank's dispatch order is expert-contiguous, so its
    // rows for expert e start at the exclusive scan of its own counts
    long long run = 0;
    for (int e = 0; e < E; ++e) {
        send_offsets[e] = (int32_t)run;
        run += mine[e];
    }
    send_offsets[E] = (int32_t)run;
    for (int h = 0; h < G; ++h) {
        long long n = 0;
        for (int e = first_expert(h, E, G); e < first_expert(h + 1, E, G); ++e) n += mine[e];
        peer_send[h] = (int32_t)n;
    }

    // receiver side: local expert j holds the rows of source 0, then source 1,
    // ...; inside a source, its own (token-ascending) order
    run = 0;
    for (int j = 0; j < el; ++j) {
        recv_offsets[j] = (int32_t)run;
        for (int s = 0; s < G; ++s) {
            recv_slot[(size_t)s * el + j] = (int32_t)run;
            run += counts_all[(size_t)s * E + e0 + j];
        }
    }
    recv_offsets[el] = (int32_t)run;
    for (int s = 0; s < G; ++s) {
        long long n = 0;
        for (int j = 0; j < el; ++j) n += counts_all[(size_t)s * E + e0 + j];
        peer_recv[s] = (int32_t)n;
    }

    // the capacity verdict on every expert of every rank: each rank reaches the
    // same answer from the same counts, so all of them skip the payload together
    for (int e = 0; e < E; ++e) {
        long long total = 0;
        for (int s = 0; s < G; ++s) total += counts_all[(size_t)s * E + e];
        if (total > capacity) {
            set_error("moe_ep_plan: expert %d would receive %lld rows, capacity %d", e, total, capacity);
            return MOE_ERR_CAPACITY;
        }
    }
    return MOE_OK;
}
