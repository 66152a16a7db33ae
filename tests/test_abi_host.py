"""Host-side checks of the C-ABI library that need no GPU: it loads, it exports every
function include/phx.h declares, and its argument checks, configuration table, config
parsing and tuner selection logic behave as documented."""
import ctypes

import pytest

from dense_gemm_04_gb300 import phx


def test_every_declared_function_is_exported():
    declared = phx.declared_functions()
    assert len(declared) >= 15
    lib = ctypes.CDLL(phx.LIB_PATH)
    missing = [f for f in declared if not hasattr(lib, f)]
    assert not missing, missing
    # the binding wraps exactly the declared set
    assert sorted(phx._SIGNATURES) == declared


def test_status_strings():
    for s in range(8):
        assert phx.status_string(s).startswith("PHX_")
    assert "unknown" in phx.status_string(99)


def test_validate_args():
    ok, bad = phx.PHX_OK, phx.PHX_ERR_INVALID
    A, B, C = 0x1000, 0x100000, 0x200000
    assert phx.validate_args(64, 64, 64, A, B, C) == ok
    assert phx.validate_args(-1, 4, 4, A, B, C) == bad
    assert phx.validate_args(4, -1, 4, A, B, C) == bad
    assert phx.validate_args(4, 4, -1, A, B, C) == bad
    assert phx.validate_args(1 << 31, 4, 4, A, B, C) == bad          # dimension too large
    assert phx.validate_args(0, 4, 4, None, None, None) == ok          # empty: nothing touched
    assert phx.validate_args(4, 0, 4, None, None, None) == ok
    assert phx.validate_args(4, 4, 0, None, None, C) == ok             # K == 0: A, B unused
    assert phx.validate_args(4, 4, 4, None, B, C) == bad               # null operand
    assert phx.validate_args(4, 4, 4, A, B, None) == bad
    assert phx.validate_args(4, 4, 4, A + 2, B, C) == bad              # not 4-byte aligned
    assert phx.validate_args(4, 4, 4, A, B, A + 32) == bad             # C overlaps A
    assert phx.validate_args(4, 4, 4, A, C - 16, C) == bad             # B overlaps C
    assert phx.validate_args(4, 4, 4, A, A, C) == ok                   # A and B may alias


def test_no_device_gives_arch_error_without_launch():
    # On a machine without a GPU, a valid call reports PHX_ERR_ARCH; an invalid one is
    # still rejected as invalid first (arguments are checked before the device).
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert phx.phx_sgemm(8, 8, 8, 1.0, 0x1000, 0x2000, 0.0, 0x3000, None) == phx.PHX_ERR_ARCH
    assert phx.phx_sgemm(-8, 8, 8, 1.0, 0x1000, 0x2000, 0.0, 0x3000, None) == phx.PHX_ERR_INVALID
    assert phx.phx_gemm_f16tc_f32acc(8, 8, 8, 1.0, 0x1000, 0x2000, 0.0, 0x1000, None) == phx.PHX_ERR_INVALID
    assert phx.phx_sgemm(0, 8, 8, 1.0, None, None, 0.0, None, None) == phx.PHX_OK


@pytest.mark.parametrize("variant", [phx.VARIANT_SGEMM, phx.VARIANT_F16TC])
def test_config_names_round_trip(variant):
    names = phx.config_names(variant)
    assert len(names) == phx.num_configs(variant) > 0
    assert len(set(names)) == len(names)
    for name in names:
        phx.set_config(variant, name)
        assert phx.get_config(variant, 4096, 4096, 4096) == name
        # keys in another order parse to the same configuration
        phx.set_config(variant, " ".join(reversed(name.split())))
        assert phx.get_config(variant, 512, 512, 512) == name
    phx.set_config(variant, None)


def test_skinny_config_name():
    for variant in (phx.VARIANT_SGEMM, phx.VARIANT_F16TC):
        names = phx.config_names(variant)
        assert names[-1] == "SKINNY" and names.count("SKINNY") == 1
        phx.set_config(variant, "  SKINNY ")
        assert phx.get_config(variant, 4096, 4096, 4096) == "SKINNY"
        for bad in ("SKINNY TILE_M=128", "SKINNY=1", "skinny"):
            with pytest.raises(phx.PhxError):
                phx.set_config(variant, bad)
        phx.set_config(variant, None)


def test_config_parse_errors():
    for spec in ("TILE_M=128", "TILE_M=128 TILE_N=128 TILE_K=7", "TILE_M=x TILE_N=1 TILE_K=1",
                 "BOGUS=1 TILE_M=128 TILE_N=128 TILE_K=8", "TILE_M=128 TILE_N=128 TILE_K=8 STAGES=9"):
        with pytest.raises(phx.PhxError) as e:
            phx.set_config(phx.VARIANT_SGEMM, spec)
        assert e.value.status == phx.PHX_ERR_CONFIG
    with pytest.raises(phx.PhxError):
        phx.set_config(phx.VARIANT_F16TC, "TILE_M=128 TILE_N=256 TILE_K=64 FMA2=1")
    with pytest.raises(phx.PhxError):
        phx.set_config(7, "TILE_M=128 TILE_N=128 TILE_K=8")
    # the pages' own example pin parses (STAGES left open)
    phx.set_config(phx.VARIANT_SGEMM, "TILE_M=128 TILE_N=128 TILE_K=8")
    assert phx.get_config(0, 64, 64, 64).startswith("TILE_M=128 TILE_N=128 TILE_K=8 ")
    phx.set_config(phx.VARIANT_SGEMM, "")


def test_default_config_follows_grid_size():
    phx.set_config(0, None)
    phx.set_config(1, None)
    big = phx.get_config(phx.VARIANT_SGEMM, 4096, 4096, 4096)
    small = phx.get_config(phx.VARIANT_SGEMM, 1024, 1024, 16384)
    skinny = phx.get_config(phx.VARIANT_SGEMM, 64, 4096, 4096)
    assert big.startswith("TILE_M=128 TILE_N=128")
    assert small.startswith("TILE_M=128 TILE_N=128")   # a small grid is split along K instead
    assert skinny.startswith("TILE_M=64 TILE_N=64")
    assert phx.get_config(phx.VARIANT_F16TC, 4096, 4096, 4096).startswith("TILE_M=256 TILE_N=256")
    # few rows of A: the skinny kernel (B streamed once) up to 48 rows (f32) and 16 (f16)
    assert phx.get_config(phx.VARIANT_SGEMM, 1, 4096, 4096) == "SKINNY"
    assert phx.get_config(phx.VARIANT_SGEMM, 48, 4096, 4096) == "SKINNY"
    assert phx.get_config(phx.VARIANT_SGEMM, 49, 4096, 4096) != "SKINNY"
    assert phx.get_config(phx.VARIANT_F16TC, 16, 4096, 4096) == "SKINNY"
    assert phx.get_config(phx.VARIANT_F16TC, 17, 4096, 4096) != "SKINNY"


def test_workspace_bytes():
    # A as M x Kp halves and B transposed as N x Kp halves, Kp = K rounded up to 8,
    # each part rounded up to 256 bytes
    def want(M, N, K):
        Kp = (K + 7) // 8 * 8
        r = lambda b: (b + 255) // 256 * 256
        return r(M * Kp * 2) + r(N * Kp * 2)
    for shape in [(4096, 4096, 4096), (4095, 4097, 4093), (1, 1, 1), (16384, 128, 4096)]:
        assert phx.f16tc_workspace_bytes(*shape) == want(*shape)


# ----------------------------------------------------------------------------------------
# The tuner's selection logic on simulated candidates ("gemm, f32", section "Tuning")
# ----------------------------------------------------------------------------------------

def test_tuner_picks_fastest():
    times = [3.0, 1.0, 2.0, 5.0, 1.5, 4.0]
    picked, launches = phx.selftest_tuner(times, noise=0.02)
    assert picked == 1
    assert launches >= 4 * len(times)


def test_tuner_skips_failing_candidates():
    times = [3.0, 1.0, 2.0, 5.0]
    picked, _ = phx.selftest_tuner(times, fail=[0, 1, 0, 0])
    assert picked == 2
    picked, _ = phx.selftest_tuner(times, fail=[1, 1, 1, 1])
    assert picked == -1


def test_tuner_second_stage_resists_drift():
    # Two finalists 3 % apart while the card slows down over the run (drift): stage 2's
    # shuffled rounds keep the faster one, whatever the order of the candidates.
    for seed in range(1, 6):
        picked, _ = phx.selftest_tuner([1.03, 1.0, 2.0], noise=0.005, drift=2e-3, seed=seed)
        assert picked == 1, seed
        picked, _ = phx.selftest_tuner([1.0, 1.03, 2.0], noise=0.005, drift=2e-3, seed=seed)
        assert picked == 0, seed


def test_tuner_cache_file_round_trip(tmp_path):
    p = tmp_path / "tune.txt"
    p.write_text("# variant M N K config\n0 4096 4096 4096 TILE_M=128 TILE_N=64 TILE_K=8 STAGES=4 FMA2=0\n"
                 "1 8192 8192 1024 TILE_M=128 TILE_N=128 TILE_K=64 STAGES=6\n")
    phx.set_config(0, None)
    phx.set_config(1, None)
    phx.tune_cache_load(str(p))
    assert phx.get_config(0, 4096, 4096, 4096) == "TILE_M=128 TILE_N=64 TILE_K=8 STAGES=4 FMA2=0"
    assert phx.get_config(1, 8192, 8192, 1024) == "TILE_M=128 TILE_N=128 TILE_K=64 STAGES=6"
    out = tmp_path / "out.txt"
    phx.tune_cache_save(str(out))
    text = out.read_text()
    assert "0 4096 4096 4096 TILE_M=128 TILE_N=64" in text
    bad = tmp_path / "bad.txt"
    bad.write_text("0 1 1 1 TILE_M=3 TILE_N=3 TILE_K=3\n")
    with pytest.raises(phx.PhxError):
        phx.tune_cache_load(str(bad))


def test_cluster_key():
    names = phx.config_names(phx.VARIANT_F16TC)
    clustered = [n for n in names if n.endswith(" CLUSTER=2")]
    assert clustered, names
    for n in clustered:
        phx.set_config(phx.VARIANT_F16TC, n)
        assert phx.get_config(phx.VARIANT_F16TC, 4096, 4096, 4096) == n
    # without the key, the pair-free configuration of the same tile is meant
    base = clustered[0].replace(" CLUSTER=2", "")
    phx.set_config(phx.VARIANT_F16TC, base)
    assert phx.get_config(phx.VARIANT_F16TC, 4096, 4096, 4096) == base
    for bad in (base + " CLUSTER=3", ):
        with pytest.raises(phx.PhxError):
            phx.set_config(phx.VARIANT_F16TC, bad)
    with pytest.raises(phx.PhxError):
        phx.set_config(phx.VARIANT_SGEMM, "TILE_M=128 TILE_N=128 TILE_K=16 CLUSTER=2")
    phx.set_config(phx.VARIANT_F16TC, None)


def test_ex_calls_check_the_op_first():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for fn in (phx.phx_sgemm_ex, phx.phx_gemm_f16tc_f32acc_ex):
        assert fn(2, 0, 8, 8, 8, 1.0, 0x1000, 0x2000, 0.0, 0x3000, None) == phx.PHX_ERR_INVALID
        assert fn(0, -1, 8, 8, 8, 1.0, 0x1000, 0x2000, 0.0, 0x3000, None) == phx.PHX_ERR_INVALID
        assert fn(1, 1, 8, 8, 8, 1.0, 0x1000, 0x2000, 0.0, 0x3000, None) == phx.PHX_ERR_ARCH
        assert fn(1, 0, 8, 8, 8, 1.0, 0x1000, 0x2000, 0.0, 0x1000, None) == phx.PHX_ERR_INVALID
        assert fn(1, 1, 0, 8, 8, 1.0, None, None, 0.0, None, None) == phx.PHX_OK


def test_binding_storage_order():
    import torch
    x = torch.zeros(5, 3)
    assert phx._operand_op(x, "A") == phx.OP_N
    assert phx._operand_op(x.t(), "A") == phx.OP_T
    assert phx._operand_op(torch.zeros(1, 4), "A") == phx.OP_N
    with pytest.raises(ValueError):
        phx._operand_op(torch.zeros(6, 6)[::2, ::2], "A")
    with pytest.raises(ValueError):
        phx._operand_op(torch.zeros(2, 3, 4), "A")


def test_f16_inputs_argument_checks():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for fn in (phx.phx_gemm_f16in_f32acc, phx.phx_gemm_f16in_f16out):
        assert fn(3, 0, 8, 8, 8, 1.0, 0x1000, 0x2000, 0.0, 0x4000, None) == phx.PHX_ERR_INVALID  # bad op
        assert fn(0, 0, 8, 8, 8, 1.0, 0x1001, 0x2000, 0.0, 0x4000, None) == phx.PHX_ERR_INVALID  # odd address
        assert fn(0, 0, 8, 8, 8, 1.0, 0x1000, 0x2000, 0.0, 0x4000, None) == phx.PHX_ERR_ARCH
        assert fn(0, 0, 0, 8, 8, 1.0, None, None, 0.0, None, None) == phx.PHX_OK
    # A (8 x 8 halves = 128 bytes) ends right where an f16 C starts: no overlap; one byte
    # earlier it overlaps
    assert phx.phx_gemm_f16in_f16out(0, 0, 8, 8, 8, 1.0, 0x1000, 0x3000, 0.0, 0x1080, None) == phx.PHX_ERR_ARCH
    assert phx.phx_gemm_f16in_f16out(0, 0, 8, 8, 8, 1.0, 0x1000, 0x3000, 0.0, 0x107E, None) == phx.PHX_ERR_INVALID
    # an f32 C must be 4-byte aligned
    assert phx.phx_gemm_f16in_f32acc(0, 0, 8, 8, 8, 1.0, 0x1000, 0x3000, 0.0, 0x4002, None) == phx.PHX_ERR_INVALID


def test_last_config_before_any_gemm():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert phx.last_config(phx.VARIANT_SGEMM) == "NONE"
    assert phx.last_config(phx.VARIANT_F16TC) == "NONE"
    with pytest.raises(phx.PhxError):
        phx.last_config(5)


def test_profile_kinds_match_the_header():
    # one name per PHX_KIND_* of include/phx.h, in order
    import re
    with open(phx.HEADER_PATH) as f:
        text = f.read()
    kinds = {m.group(1): int(m.group(2)) for m in re.finditer(r"PHX_KIND_([A-Z0-9_]+)\s*=\s*(\d+)", text)}
    num = int(re.search(r"PHX_NUM_KINDS\s*=\s*(\d+)", text).group(1))
    assert len(phx.KIND_NAMES) == num == len(kinds)
    for name, idx in kinds.items():
        assert phx.KIND_NAMES[idx] == name.lower(), (name, idx)
