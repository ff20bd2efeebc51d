"""Host-side helpers of bench.py that need no GPU."""
import torch

import bench


def test_tile_scales_layout():
    # the tiled layout gemm_mxfp8_tiled takes, written out element by element
    import gemm_inputs as gi
    rows, K = 300, 32 * 9          # ragged rows and a partial block group
    nb = (K + 31) // 32
    g = torch.Generator().manual_seed(1)
    sf = torch.randint(0, 255, (rows, 16), dtype=torch.uint8, generator=g)
    out = gi.tile_scales(sf, rows, K)
    G = (nb + 3) // 4
    assert out.numel() == (rows + 127) // 128 * G * 512
    for r in range(384):
        for b in range(4 * G):
            off = 512 * ((r // 128) * G + b // 4) + 16 * (r % 32) + 4 * ((r % 128) // 32) + b % 4
            want = int(sf[r, b]) if r < rows and b < nb else 0
            assert int(out[off]) == want, (r, b)


def test_blocked_scales_layout():
    # cuBLASLt's block-scaled layout, written out element by element: a 128-row x
    # 4-block tile is 512 bytes, tiles ordered row-block major; inside a tile, row
    # r's byte for block c sits at 16*(r % 32) + 4*(r // 32) + c.
    rows, K = 200, 8 * 32 * 3          # ragged rows, 24 blocks: 6 groups of 4
    nb = K // 32
    g = torch.Generator().manual_seed(0)
    sf = torch.randint(0, 255, (rows, 32), dtype=torch.uint8, generator=g)
    out = bench.blocked_scales(sf, rows, K).view(torch.uint8).flatten()
    R, C = 256, (nb + 3) // 4 * 4
    assert out.numel() == R * C
    for r in range(R):
        for b in range(C):
            tile = (r // 128) * (C // 4) + b // 4
            rr = r % 128
            off = tile * 512 + 16 * (rr % 32) + 4 * (rr // 32) + b % 4
            want = int(sf[r, b]) if r < rows and b < nb else 0
            assert int(out[off]) == want, (r, b)


def test_tensor_peak_choice():
    # the sustained (power-capped, seconds-long) peak only for a region that
    # is itself seconds long and saw the power cap; a short burst otherwise
    capped = {"reasons": ["sw_power_cap"]}
    assert bench.tensor_peak_choice(0.019, {"reasons": []})[0] == "burst"
    assert bench.tensor_peak_choice(0.019, capped)[0] == "burst"
    assert bench.tensor_peak_choice(5.0, {"reasons": []})[0] == "burst"
    assert bench.tensor_peak_choice(5.0, None)[0] == "burst"
    assert bench.tensor_peak_choice(1.2, capped)[0] == "sustained"


def test_clock_sampler_takes_the_median_under_load():
    # nvidia-smi rows as the sampler queries them: index, clocks.sm, clocks.max.sm,
    # power.draw, reasons.active, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap,
    # power.limit.  Idle samples (boost clock, low power) sit around the loaded ones.
    rows = [
        "0, 2070, 2070, 180.5, 0x0, Not Active, Not Active, Not Active, Not Active, 1400.00",
        "0, 1665, 2070, 1210.0, 0x0, Not Active, Not Active, Not Active, Not Active, 1400.00",
        "0, 1650, 2070, 1302.4, 0x4, Not Active, Not Active, Not Active, Active, 1400.00",
        "0, 1680, 2070, 1190.2, 0x0, Not Active, Not Active, Not Active, Not Active, 1400.00",
        "0, 2070, 2070, 175.0, 0x0, Not Active, Not Active, Not Active, Not Active, 1400.00",
        "garbage line",
    ]

    class FakeProc:
        def terminate(self):
            pass

        def communicate(self, timeout=None):
            return "\n".join(rows) + "\n", ""

    s = bench.ClockSampler(0)
    s.proc = FakeProc()
    clk = s.stop()
    assert clk["samples"] == 5 and clk["samples_under_load"] == 3
    assert clk["sm_mhz"] == 1665.0
    assert clk["sm_mhz_all_samples"] == 1680.0
    assert clk["sm_max_mhz"] == 2070.0
    assert clk["reasons"] == ["sw_power_cap"]
    assert clk["active_masks"] == ["0x0", "0x4"]
    assert clk["power_w_max"] == 1302.4
    # no sample under load: the median over all of them
    rows[1:4] = []
    s.proc = FakeProc()
    clk = s.stop()
    assert clk["samples_under_load"] == 0 and clk["sm_mhz"] == 2070.0


def test_clock_sampler_prefers_samples_inside_the_timed_region():
    # the same fields plus the host timestamp; power.draw is an average that
    # a short region never lifts, so only the timestamps tell which samples
    # fall inside it
    import datetime
    t = [datetime.datetime(2026, 1, 2, 3, 4, 5, 100000 * i) for i in range(6)]
    f = [x.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3] for x in t]
    rows = [
        f"0, 2070, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active, 1400.00, {f[0]}",
        f"0, 1710, 2070, 160.0, 0x0, Not Active, Not Active, Not Active, Not Active, 1400.00, {f[2]}",
        f"0, 1690, 2070, 170.0, 0x0, Not Active, Not Active, Not Active, Not Active, 1400.00, {f[3]}",
        f"0, 1700, 2070, 170.0, 0x0, Not Active, Not Active, Not Active, Not Active, 1400.00, {f[4]}",
        f"0, 2070, 2070, 175.0, 0x0, Not Active, Not Active, Not Active, Not Active, 1400.00, {f[5]}",
    ]

    class FakeProc:
        def terminate(self):
            pass

        def communicate(self, timeout=None):
            return "\n".join(rows) + "\n", ""

    s = bench.ClockSampler(0)
    s.proc = FakeProc()
    clk = s.stop((t[1].timestamp(), t[4].timestamp() + 0.01))
    assert clk["samples"] == 5 and clk["samples_under_load"] == 0
    assert clk["samples_in_region"] == 3 and clk["sm_mhz"] == 1700.0
    s.proc = FakeProc()
    clk = s.stop()   # no window: nothing inside, the median over all samples
    assert clk["samples_in_region"] == 0 and clk["sm_mhz"] == 1710.0
