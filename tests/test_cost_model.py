"""The cost model against the numbers the pages print (tests/golden/pages_numbers.txt), and
the per-kernel byte counts against hand counts.  CPU only."""
import os

import pytest

from depth_wise_softmax_block_b300 import cost as C

GOLD = os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.txt")
MiB, GiB = 2 ** 20, 2 ** 30


def _load():
    rows = {}
    for line in open(GOLD, encoding="utf-8"):
        if not line.strip() or line.startswith("#"):
            continue
        key, val, tol, _cite = [x.strip() for x in line.split("|", 3)]
        rows[key] = (float(val), float(tol))
    return rows


COMPUTED = {
    "n_pairs_L122": lambda: C.n_pairs(122),
    "full_fwd_gflop_L122_d7168": lambda: C.full_fwd_flops_per_token(122, 7168) / 1e9,
    "params_2Ld_million": lambda: 2 * 122 * 7168 / 1e6,
    "full_train_gflop_L122": lambda: 3 * C.full_fwd_flops_per_token(122, 7168) / 1e9,
    "full_history_GB_T32K_L128": lambda: C.full_history_bytes(1, 32768, 128, 7168) / 1e9,
    "full_history_GB_8way": lambda: C.full_history_bytes(1, 32768, 128, 7168) / 8 / 1e9,
    "decode_depth_state_MiB": lambda: 123 * 7168 * 2 / MiB,
    "hidden_state_MiB_M4096": lambda: 4096 * 7168 * 2 / MiB,
    "full_history_GiB_123": lambda: 123 * (4096 * 7168 * 2) / GiB,
    "block_history_MiB_8": lambda: 8 * 4096 * 7168 * 2 / MiB,
    "block_history_MiB_9": lambda: 9 * 4096 * 7168 * 2 / MiB,
    "block_cache_GB_128K_N8": lambda: C.block_cache_bytes(1, 8, 131072, 7168) / 1e9,
    "block_cache_GB_P8": lambda: C.block_cache_bytes(1, 8, 131072, 7168, P=8) / 1e9,
    "block_cache_GB_P8_chunk16K_max": lambda: C.block_cache_bytes(1, 8, 16384, 7168, P=8) / 1e9,
    "io_standard_d": lambda: C.io_per_layer_standard(1),
    "io_full_two_phase_d": lambda: C.io_per_layer_full_two_phase(16, 8, 1),
    "io_block_two_phase_d": lambda: C.io_per_layer_block_two_phase(16, 8, 1),
    "io_mhc_d_coeff": lambda: C.io_per_layer_mhc(4, 1000) // 1000,
    "io_mhc_scalar": lambda: C.io_per_layer_mhc(4, 1000) % 1000,
    "pp_comm_naive_P4_V2": lambda: C.pp_comm_naive(4, 2),
    "pp_comm_cached_P4_V2": lambda: C.pp_comm_cached(4, 2),
}


@pytest.mark.parametrize("key", sorted(COMPUTED))
def test_pages_numbers(key):
    val, tol = _load()[key]
    got = COMPUTED[key]()
    if key.endswith("_max"):
        assert got < val
    elif tol == 0:
        assert got == val
    else:
        assert abs(got - val) <= tol * abs(val), (key, got, val)


def test_every_golden_row_checked():
    assert set(_load()) == set(COMPUTED)


def test_kernel_bytes_hand_counts():
    d, E = 7168, 2
    assert C.phase1_bytes(9, 24, d, E) == 33 * d * E + 96
    assert C.phase2_bytes(d, E, False, False) == 2 * d * E
    assert C.phase2_bytes(d, E, True, False) == 3 * d * E + 4
    assert C.phase2_bytes(d, E, True, True) == 5 * d * E + 4
    st = C.block_step_bytes(9, 24, d, E, final_sources=10)
    assert st.phase1 == 33 * d * E + 4 * 24          # o and lse; m is not written
    assert st.phase2 == 2 * d * E + (3 * d * E + 4) + 22 * (5 * d * E + 4)
    assert st.close == 3 * d * E
    assert st.final == 11 * d * E
    assert C.phase1_flops(9, 24, d) == 2 * (2 * 24 * 9 * d + 9 * d)


def test_head_statistics_bytes():
    """With H heads every 4-byte statistic is kept per head: phase 1 writes S*H lse values per
    token, phase 2 reads H."""
    d, E = 7168, 2
    assert C.phase1_bytes(9, 24, d, E, heads=16) - C.phase1_bytes(9, 24, d, E) == 4 * 24 * 15
    assert C.phase2_bytes(d, E, True, True, heads=16) - C.phase2_bytes(d, E, True, True) == 4 * 15
    assert C.phase2_bytes(d, E, False, False, heads=16) == C.phase2_bytes(d, E, False, False)
    b1 = C.block_step_bytes(9, 24, d, E, 10)
    b16 = C.block_step_bytes(9, 24, d, E, 10, heads=16)
    assert b16.phase1 - b1.phase1 == 4 * 24 * 15
    assert b16.phase2 - b1.phase2 == 23 * 4 * 15      # 23 calls read the partial's lse
    assert (b16.close, b16.final) == (b1.close, b1.final)


def test_walk_bytes_hand_count():
    """The walk bench's bytes per depth walk: block n (1-based) runs phase 1 over n sources for
    its S_n sublayers, S_n phase-2 calls and the close; then the final aggregation over all
    closed blocks and the embedding.  The decode and prefill-chunk walks (186 sublayers in
    7 x 24 + 18, bf16) and the tiny fp32 walk (8 sublayers in 2 x 4)."""
    import bench
    from synth import inputs as I
    for wl, E, blocks in [(I.DECODE_BF16, 2, [24] * 7 + [18]),
                          (I.PREFILL_CHUNK_BF16, 2, [24] * 7 + [18]),
                          (I.TINY_BLOCK_F32, 4, [4, 4])]:
        d, T = wl.d, wl.T
        want = 0
        for n, Sn in enumerate(blocks, start=1):
            want += (n + Sn) * d * E + 4 * Sn              # phase 1: sources, o; lse
            want += 2 * d * E                              # sublayer 1: read o, write y
            want += 3 * d * E + 4                          # sublayer 2: o, lse, v_1; write y
            want += (Sn - 2) * (5 * d * E + 4)             # sublayers 3..: fused update
            want += 3 * d * E                              # close
        nf = len(blocks) + 1
        want += (nf + 1) * d * E                           # final: read all slots, write 1
        assert bench.walk_bytes(wl) == want * T, wl.name


def test_traffic_lookup_matches_kernel_sources(tmp_path, monkeypatch):
    """A committed DRAM-traffic capture is used only for the sources it measured: the entry's
    hash must equal the hash of the kernel's own files."""
    import json
    import bench
    prof = tmp_path / "profiles"
    prof.mkdir()
    good = {"phase2_fused": {"src_hash": bench.kernel_hash("phase2_fused"),
                             "bytes_per_launch": 123.0},
            "phase1": {"src_hash": "0" * 16, "bytes_per_launch": 456.0}}
    (prof / "dram_traffic_longctx_T4096.json").write_text(json.dumps(good))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("phase2_fused") == 123.0
    assert bench.traffic_for("phase1") is None                 # stale entry
    assert bench.traffic_for("final") is None                  # no entry
    assert bench.traffic_for("phase2_fused", heads=16) is None  # no file for 16 heads
