"""Plan rules restated from their definitions, for the tests that check the plans' choices."""


def e4m3_tile_rule(M, N, K, f32, units=76):
    """The e4m3 pair tile-width rule: column share x round share (0.89 under stream-K), x 0.93 for
    224 or, for 256, the tile boundary of 3.8 k-blocks per tile after a unit's first; 224 must win
    by 5 %."""
    tiles_m, kb = -(-M // 256), -(-K // 128)

    def eff(bn):
        tn = -(-N // bn)
        tiles = tiles_m * tn
        rounds = -(-tiles // units)
        sk = f32 and kb >= 64 and tiles >= units and tiles % units != 0 and tiles < 4 * units
        e = N / (tn * bn) * (0.89 if sk else tiles / (rounds * units))
        return e * (0.93 if bn == 224 else 1.0 - 3.8 / kb * (1.0 - 1.0 / rounds))
    return 224 if eff(224) > 1.05 * eff(256) else 256
