"""The benchmark's byte and flop models, against the sizes the workloads fix
(compulsory traffic: read x, dt, B, C, A, D and the initial state once, write
y in bf16 and the final state once; flops of the chunked algorithm with full
Q x Q tiles)."""
import pytest

import bench
import ssd_inputs as si

# (workload, compulsory MB, GFLOP)
EXPECTED = [
    ("mamba2_130m", 58.1, 8.24),
    ("mamba2_2p7b", 183.8, 27.15),
    ("long_16k", 212.9, 32.68),
    ("wide_head", 706.7, 160.0),
    ("wide_head_q128", 706.7, 180.9),
]


@pytest.mark.parametrize("name,mb,gflop", EXPECTED)
def test_compulsory_bytes_and_flops(name, mb, gflop):
    cfg = si.CONFIGS[name]
    assert bench.compulsory_bytes(cfg) / 1e6 == pytest.approx(mb, abs=0.05)
    assert bench.chunked_flops(cfg) / 1e9 == pytest.approx(gflop, rel=2e-3)


def test_compulsory_bytes_by_hand():
    # 130M layer: x 4*2048*24*64*2, dt 4*2048*24*2, B and C 2*(4*2048*128*2),
    # A and D 2*24*4, y 4*2048*24*64*2, final 4*24*64*128*4
    cfg = si.CONFIGS["mamba2_130m"]
    want = (4 * 2048 * 24 * 64 * 2 + 4 * 2048 * 24 * 2 + 2 * 4 * 2048 * 128 * 2 + 2 * 24 * 4
            + 4 * 2048 * 24 * 64 * 2 + 4 * 24 * 64 * 128 * 4)
    assert bench.compulsory_bytes(cfg) == want


def test_kernel_bytes_cover_the_compulsory_traffic():
    # every byte the operation must move is counted by one of the three
    # tensor-core kernels (they also move intermediates: packs, segment states)
    for name, _, _ in EXPECTED:
        cfg = si.CONFIGS[name]
        k = sum(bench.KERNEL_BYTES(cfg, n) for n in ("cb_mask_tc", "seg_state_tc", "chunk_scan_tc"))
        assert k >= bench.compulsory_bytes(cfg)
