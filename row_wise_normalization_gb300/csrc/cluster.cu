// Cluster-split kernels: one row over 2..16 CTAs, statistics exchanged through
// distributed shared memory.
#include "rn_cluster.cuh"

namespace rn {

template <int OP, bool AL>
const ClusterEntry* cluster_pick(int slots, int threads, int cl) {
    if (threads == 256) {
        // 4 quads a thread only on 2 CTAs: a wider cluster of 4 quads holds
        // what half as many CTAs of 8 quads hold, and the planner takes those
        if (cl == 2 && slots == 4) return &ClusterInst<OP, 4, 256, 2, AL>::entry;
#define RN_CL(CLV) \
    if (cl == CLV) {                                                            \
        if (slots == 6) return &ClusterInst<OP, 6, 256, CLV, AL>::entry;       \
        if (slots == 8) return &ClusterInst<OP, 8, 256, CLV, AL>::entry;       \
    }
        RN_CL(2) RN_CL(4) RN_CL(8) RN_CL(16)
#undef RN_CL
        return nullptr;
    }
    if (cl != 16 || slots != 8) return nullptr;
    if (threads == 512) return &ClusterInst<OP, 8, 512, 16, AL>::entry;
    if (threads == 1024) return &ClusterInst<OP, 8, 1024, 16, AL>::entry;
    return nullptr;
}

const ClusterEntry* cluster_entry(int op, int slots, int threads, int cl, bool al) {
    if (op == OP_LN)
        return al ? cluster_pick<OP_LN, true>(slots, threads, cl)
                  : cluster_pick<OP_LN, false>(slots, threads, cl);
    return al ? cluster_pick<OP_RMS, true>(slots, threads, cl)
              : cluster_pick<OP_RMS, false>(slots, threads, cl);
}

}  // namespace rn
