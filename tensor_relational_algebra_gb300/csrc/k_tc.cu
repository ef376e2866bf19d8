// Tensor-core (tcgen05 / TMEM / TMA) join + aggregate for BF16 sum-of-products.
#include "plan.h"

namespace tra {

struct TcPlan {};

bool tc_plan(Plan*) { return false; }
void tc_free(TcPlan* t) { delete t; }
int tc_execute(const Plan&, const void*, const void*, void*, cudaStream_t) {
    return fail(TRA_ERR_UNSUPPORTED, "tensor-core path not available");
}

}  // namespace tra
