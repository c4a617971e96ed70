// Host probe of the tile kernel's work decomposition, for tests/test_plan_host.py.
//
// Reads lines "M N K BM BN BK resident streamk" from stdin and prints, per
// line, the plan_launch() result: "ok tiles_m tiles_n iters_per_tile dp_tiles
// sk_tiles sk_ctas sk_base sk_extra grid slots group_m spec", spec being the
// size-specialized instance find_specialized_plan() names for that launch
// with the default configuration of its tiles (-1: none).  plan_launch is the
// constexpr function that the host API and the size-specialized kernels both
// evaluate, so this is the decomposition the GPU runs.
#include <cstdio>

#include "sgemm_plan.h"

int main() {
  long long M, N, K, resident;
  int bm, bn, bk, streamk;
  while (std::scanf("%lld %lld %lld %d %d %d %lld %d", &M, &N, &K, &bm, &bn, &bk, &resident,
                    &streamk) == 8) {
    const gb300::LaunchPlan p = gb300::plan_launch(M, N, K, bm, bn, bk, resident, streamk != 0);
    // The size-specialized instance the host would take for this launch with
    // the default configuration of these tiles (0: 128 x 256, 3: 128 x 128).
    const int cfg = bn == 256 ? 0 : 3;
    const int spec = gb300::find_specialized_plan(cfg, M, N, K, bm, bn, bk, resident, p.sc, p.grid);
    std::printf("%d %d %d %d %d %d %d %d %d %lld %lld %d %d\n", p.ok ? 1 : 0, p.sc.tiles_m,
                p.sc.tiles_n, p.sc.iters_per_tile, p.sc.dp_tiles, p.sc.sk_tiles, p.sc.sk_ctas,
                p.sc.sk_base, p.sc.sk_extra, static_cast<long long>(p.grid),
                static_cast<long long>(p.slots), p.sc.group_m, spec);
  }
  return 0;
}
