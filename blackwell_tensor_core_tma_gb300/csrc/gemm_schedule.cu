// Test hook (declared in include/gb300gemm_testing.h): the kernels' work schedule, run on
// the host.  The persistent GEMM and chain kernels walk their pieces with WorkIter and
// ChainIter (gemm_kernel.cuh), plain integer code compiled for host and device alike; this
// entry point lists one unit's pieces so that the schedule's coverage can be checked
// without a device.
#include "gemm_kernel.cuh"

extern "C" gemm_status gemm_testing_schedule(int chain, int tiles_m, int tiles_n, int group_m, int num_kb,
                                             int splits, int sk_dp_tiles, int sk_units, int unit, int units,
                                             int *out, int max_pieces, int *n_pieces) {
    using namespace gb300;
    if (!out || !n_pieces || max_pieces < 0 || tiles_m <= 0 || num_kb <= 0 || units <= 0 || unit < 0 ||
        unit >= units || sk_dp_tiles < 0 || sk_units < 0)
        return GEMM_ERR_INVALID_ARG;
    const bool sk = sk_units > 0;
    if (sk && (sk_units != units || sk_dp_tiles % units != 0)) return GEMM_ERR_INVALID_ARG;
    int n = 0;
    Work w;
    auto emit = [&]() {
        if (n < max_pieces) {
            int *o = out + 6 * n;
            o[0] = w.tm;
            o[1] = w.tn;
            o[2] = w.kb0;
            o[3] = w.kb1;
            o[4] = w.role;
            o[5] = w.slot;
        }
        ++n;
    };
    if (chain) {
        if (sk && sk_dp_tiles >= tiles_m) return GEMM_ERR_INVALID_ARG;
        ChainParams cp{};
        cp.tiles = tiles_m;
        cp.num_kb1 = num_kb;
        cp.sk = sk;
        cp.sk_dp_tiles = sk_dp_tiles;
        cp.sk_units = sk_units;
        ChainIter it(cp, unit, units);
        while (it.next(cp, w)) emit();
    } else {
        if (tiles_n <= 0 || group_m <= 0 || splits <= 0 || splits > num_kb || (sk && splits != 1) ||
            (sk && sk_dp_tiles >= tiles_m * tiles_n))
            return GEMM_ERR_INVALID_ARG;
        KParams kp{};
        kp.tiles_m = tiles_m;
        kp.tiles_n = tiles_n;
        kp.num_tiles = tiles_m * tiles_n;
        kp.group_m = group_m;
        kp.num_kb = num_kb;
        kp.splits = splits;
        kp.sk = sk;
        kp.sk_dp_tiles = sk_dp_tiles;
        kp.sk_units = sk_units;
        WorkIter it(kp, unit, units);
        while (it.next(kp, w)) emit();
    }
    *n_pieces = n;
    return GEMM_OK;
}
