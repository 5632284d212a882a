// Bounds-check hooks that vanish from normal builds token for token.
//
// `cond CTP_AND_IN(i, n, site)` appends `&& ctp_in(i, n, site)` to a condition in
// bounds-checked builds (-DCTP_CHECK: index i tested against extent n, counted
// and the access skipped when outside) and nothing otherwise;
// CTP_CHECKED_LDG(p, i, n, site) is `__ldg(p)` normally and the tested load
// (0 when outside) in checked builds.
#pragma once

#include "ctp_internal.h"

namespace ctp {

// Access sites of the analytical operators and the geometry gradients.
constexpr int kSiteFdkGather = 30, kSiteFdkStore = 31, kSiteFdkScatterLoad = 32,
              kSiteFdkScatter = 33;
constexpr int kSiteGeomRayLoad = 40, kSiteGeomColumnLoad = 41, kSiteGeomSinoLoad = 42,
              kSiteGeomOut = 43;

}  // namespace ctp

#ifdef CTP_CHECK
#define CTP_AND_IN(i, n, site) &&::ctp::ctp_in((long long)(i), (long long)(n), (site))
#define CTP_CHECKED_LDG(p, i, n, site) \
    (::ctp::ctp_in((long long)(i), (long long)(n), (site)) ? __ldg(p) : 0.0f)
#else
#define CTP_AND_IN(i, n, site)
#define CTP_CHECKED_LDG(p, i, n, site) __ldg(p)
#endif
