// uvw.cu -- placeholder, replaced by the streaming uvw radial convolution.
#include "internal.h"
namespace cgtp {
cgtp_status uvw_create(cgtp_plan_s*) { return fail(CGTP_EUNSUPPORTED, "uvw not built yet"); }
void uvw_destroy(cgtp_plan_s*) {}
cgtp_status uvw_forward(const cgtp_plan_s*, const cgtp_graph_s*, const void*, const void*, const void*,
                        const void*, void*, void*) { return fail(CGTP_EUNSUPPORTED, "uvw"); }
cgtp_status uvw_backward(const cgtp_plan_s*, const cgtp_graph_s*, const void*, const void*, const void*,
                         const void*, const void*, void*, void*, void*, void*, void*) {
  return fail(CGTP_EUNSUPPORTED, "uvw");
}
}  // namespace cgtp
