// Forward entry: exact softmax attention O = softmax(scale * Q K^T
// [bottom-right causal mask]) V with the natural-log LSE per query row
// (FFPA docs, "CuTe-DSL Backend" page, "Hard constraints"; "Varlen (packed
// THD) API"). The work runs in the cluster-exchange kernel (xchg.cu) with
// the forward operation: each CTA of a cluster scores its own key tiles,
// the CTAs agree on the running row maximum and exchange P, and every CTA
// accumulates its own head-dim slab of O.
#include "kernels.h"

namespace ffpa {

cudaError_t launch_fwd(const FwdArgs& f, cudaStream_t s)
{
    XArgs a{};
    a.pb = f.pb;
    a.bf16 = f.bf16;
    a.q = f.q;
    a.k = f.k;
    a.v = f.v;
    a.o = f.o;
    a.lse = f.lse;
    a.ctl = f.ctl;
    return launch_xchg(XOP_FWD, a, s);
}

}  // namespace ffpa
