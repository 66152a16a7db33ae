"""Host-side checks of the C-ABI library that need no GPU: it loads, it exports every
function include/phx.h declares, and its argument checks, configuration table, config
parsing and tuner selection logic behave as documented."""
import ctypes
import os

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
    assert skinny.startswith("TILE_M=64 TILE_N=128")
    assert phx.get_config(phx.VARIANT_F16TC, 4096, 4096, 4096).startswith("TILE_M=256 TILE_N=256")
    # small problems: smaller tiles give more SMs work (152 SMs assumed without a GPU)
    assert phx.get_config(phx.VARIANT_SGEMM, 512, 512, 1024).startswith("TILE_M=128 TILE_N=64 TILE_K=8 ")
    assert phx.get_config(phx.VARIANT_SGEMM, 1024, 256, 256).startswith("TILE_M=128 TILE_N=64 TILE_K=8 ")
    # ... and smaller f32 problems, or 64 rows against a B that L2 holds, the skinny kernel
    assert phx.get_config(phx.VARIANT_SGEMM, 512, 512, 512) == "SKINNY"
    assert phx.get_config(phx.VARIANT_SGEMM, 256, 256, 256) == "SKINNY"
    assert phx.get_config(phx.VARIANT_SGEMM, 64, 2048, 2048) == "SKINNY"
    assert phx.get_config(phx.VARIANT_SGEMM, 64, 4096, 4096) != "SKINNY"
    assert phx.get_config(phx.VARIANT_SGEMM, 768, 768, 768) != "SKINNY"
    # fewer than 128 rows, many columns: 64 x 128 tiles up to 64 rows, 128 x 128 above
    assert phx.get_config(phx.VARIANT_SGEMM, 64, 4096, 4096).startswith("TILE_M=64 TILE_N=128 TILE_K=16 ")
    assert phx.get_config(phx.VARIANT_SGEMM, 96, 4096, 4096).startswith("TILE_M=128 TILE_N=128 TILE_K=16 ")
    assert phx.get_config(phx.VARIANT_SGEMM, 4096, 64, 4096).startswith("TILE_M=128 TILE_N=64 TILE_K=16 ")
    assert phx.get_config(phx.VARIANT_SGEMM, 4096, 96, 4096).startswith("TILE_M=128 TILE_N=128 TILE_K=16 ")
    assert phx.get_config(phx.VARIANT_SGEMM, 1024, 1024, 1024).startswith("TILE_M=128 TILE_N=128")
    assert phx.get_config(phx.VARIANT_F16TC, 512, 512, 512).startswith("TILE_M=128 TILE_N=128")
    assert phx.get_config(phx.VARIANT_F16TC, 256, 256, 256).endswith(" CONVERT_A=1 CONVERT_B=1")
    assert phx.get_config(phx.VARIANT_F16TC, 1024, 1024, 1024).startswith("TILE_M=128 TILE_N=128")
    assert phx.get_config(phx.VARIANT_F16TC, 2048, 2048, 2048).startswith("TILE_M=128 TILE_N=256")
    # ... but a grid split along K keeps the 2-SM tile
    assert phx.get_config(phx.VARIANT_F16TC, 1024, 1024, 16384).startswith("TILE_M=256 TILE_N=256")
    # few columns, many rows: the kernel that rounds A itself, its tile as wide as N needs
    for n, tile_n in ((64, 64), (100, 128), (128, 128), (200, 256), (256, 256)):
        cfg = phx.get_config(phx.VARIANT_F16TC, 16384, n, 4096)
        assert cfg.startswith(f"TILE_M=128 TILE_N={tile_n} ") and cfg.endswith(" CONVERT_A=1"), (n, cfg)
    assert "CONVERT_A" not in phx.get_config(phx.VARIANT_F16TC, 16384, 257, 4096)
    assert phx.get_config(phx.VARIANT_F16TC, 4096, 128, 4096).endswith(" CONVERT_A=1")  # K split
    assert "CONVERT_A" not in phx.get_config(phx.VARIANT_F16TC, 4096, 128, 1024)  # too short to split
    assert phx.get_config(phx.VARIANT_F16TC, 8192, 64, 2048).endswith(" CONVERT_A=1")
    assert "CONVERT_A" not in phx.get_config(phx.VARIANT_F16TC, 2048, 128, 2048)  # A below 2^23
    assert "CONVERT_A" not in phx.get_config(phx.VARIANT_F16TC, 1024, 128, 4096)  # too few rows
    # few rows, many columns: the kernel that rounds B itself (up to 16 rows: the skinny kernel)
    for m in (9, 16, 17, 64, 256):
        assert phx.get_config(phx.VARIANT_F16TC, m, 4096, 4096).endswith(" CONVERT_B=1")
    assert phx.get_config(phx.VARIANT_F16TC, 8, 4096, 4096) == "SKINNY"
    assert phx.get_config(phx.VARIANT_F16TC, 16, 1024, 1024) == "SKINNY"       # a small B
    assert "CONVERT" not in phx.get_config(phx.VARIANT_F16TC, 64, 1024, 1024)
    assert "CONVERT" not in phx.get_config(phx.VARIANT_F16TC, 257, 4096, 4096)
    with pytest.raises(phx.PhxError):
        phx.set_config(phx.VARIANT_SGEMM, "TILE_M=128 TILE_N=128 TILE_K=16 CONVERT_B=1")
    # the f32 variant has no such key
    with pytest.raises(phx.PhxError):
        phx.set_config(phx.VARIANT_SGEMM, "TILE_M=128 TILE_N=128 TILE_K=16 CONVERT_A=1")
    # few rows of A: the skinny kernel (B streamed once) up to 48 rows (f32) and 16 (f16), or 8
    # (f16) where B is large enough for the kernel that rounds B itself
    assert phx.get_config(phx.VARIANT_SGEMM, 1, 4096, 4096) == "SKINNY"
    assert phx.get_config(phx.VARIANT_SGEMM, 48, 4096, 4096) == "SKINNY"
    assert phx.get_config(phx.VARIANT_SGEMM, 49, 4096, 4096) != "SKINNY"
    assert phx.get_config(phx.VARIANT_F16TC, 8, 4096, 4096) == "SKINNY"
    assert phx.get_config(phx.VARIANT_F16TC, 9, 4096, 4096) != "SKINNY"
    assert phx.get_config(phx.VARIANT_F16TC, 16, 2048, 2048) == "SKINNY"
    assert phx.get_config(phx.VARIANT_F16TC, 17, 2048, 2048) != "SKINNY"
    # few columns against many rows (A of 2^22 elements or more): the skinny kernel, on the
    # transposed product
    assert phx.get_config(phx.VARIANT_SGEMM, 4096, 16, 4096) == "SKINNY"
    assert phx.get_config(phx.VARIANT_SGEMM, 4096, 17, 4096) != "SKINNY"
    assert phx.get_config(phx.VARIANT_F16TC, 4096, 4, 4096) == "SKINNY"
    assert phx.get_config(phx.VARIANT_F16TC, 2048, 8, 2048) == "SKINNY"
    assert phx.get_config(phx.VARIANT_F16TC, 4096, 8, 4096).endswith(" CONVERT_A=1")
    assert phx.get_config(phx.VARIANT_F16TC, 16384, 4, 4096).endswith(" CONVERT_A=1")
    assert phx.get_config(phx.VARIANT_SGEMM, 16384, 16, 4096) == "SKINNY"
    assert phx.get_config(phx.VARIANT_SGEMM, 1000, 4, 8192) != "SKINNY"    # fewer than 1024 rows
    assert phx.get_config(phx.VARIANT_SGEMM, 4096, 4, 512) != "SKINNY"     # A below 2^22


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


def test_tuner_cache_is_keyed_by_device(tmp_path):
    tag = phx.device_tag()          # "none" on a host without a GPU
    assert tag == "none" or ":" in tag
    other = "OTHER_GPU:10" if tag != "OTHER_GPU:10" else "OTHER_GPU:11"
    p = tmp_path / "tune.txt"
    p.write_text("# device variant M N K config\n"
                 f"{tag} 0 4096 4096 4096 TILE_M=128 TILE_N=64 TILE_K=8 STAGES=4 FMA2=0\n"
                 f"{tag} 1 8192 8192 1024 TILE_M=128 TILE_N=128 TILE_K=64 STAGES=6\n"
                 f"{other} 0 2048 2048 2048 TILE_M=64 TILE_N=64 TILE_K=8 STAGES=4\n")
    phx.set_config(0, None)
    phx.set_config(1, None)
    default_2048 = phx.get_config(0, 2048, 2048, 2048)
    phx.tune_cache_load(str(p))
    assert phx.get_config(0, 4096, 4096, 4096) == "TILE_M=128 TILE_N=64 TILE_K=8 STAGES=4 FMA2=0"
    assert phx.get_config(1, 8192, 8192, 1024) == "TILE_M=128 TILE_N=128 TILE_K=64 STAGES=6"
    # another GPU's entry is kept but never applied here
    assert phx.get_config(0, 2048, 2048, 2048) == default_2048
    out = tmp_path / "out.txt"
    phx.tune_cache_save(str(out))
    text = out.read_text()
    assert f"{tag} 0 4096 4096 4096 TILE_M=128 TILE_N=64" in text
    assert f"{other} 0 2048 2048 2048 TILE_M=64 TILE_N=64" in text
    for bad_line in ("0 4096 4096 4096 TILE_M=128 TILE_N=64 TILE_K=8\n",      # no device tag
                     f"{tag} 0 1 1 1 TILE_M=3 TILE_N=3 TILE_K=3\n"):         # no such config
        bad = tmp_path / "bad.txt"
        bad.write_text(bad_line)
        with pytest.raises(phx.PhxError):
            phx.tune_cache_load(str(bad))


def _fresh_process(code, env):
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    full_env = dict(os.environ, **env)
    return subprocess.run([sys.executable, "-c", code], cwd=root, env=full_env,
                          capture_output=True, text=True, timeout=300)


def test_unparsable_env_pin_is_an_error_not_ignored():
    code = ("from dense_gemm_04_gb300 import phx\n"
            "try:\n"
            "    phx.get_config(0, 512, 512, 512)\n"
            "    print('NO ERROR')\n"
            "except phx.PhxError as e:\n"
            "    print('ERR', e.status)\n"
            "print('F16', phx.get_config(1, 512, 512, 512))\n"
            "phx.set_config(0, None)\n"
            "print('AFTER', phx.get_config(0, 512, 512, 512))\n")
    r = _fresh_process(code, {"PHX_CONFIG_SGEMM": "TILE_M=3 TILE_N=3 TILE_K=3"})
    assert r.returncode == 0, r.stderr
    lines = r.stdout.splitlines()
    assert lines[0] == f"ERR {phx.PHX_ERR_CONFIG}", r.stdout
    assert lines[1].startswith("F16 TILE_M="), r.stdout       # the other variant is unaffected
    assert lines[2] == "AFTER SKINNY", r.stdout               # phx_set_config replaces the pin
    assert "PHX_CONFIG_SGEMM" in r.stderr                     # logged, whatever PHX_LOG says


def test_tune_cache_env_file_is_read_at_first_use(tmp_path):
    p = tmp_path / "cache.txt"
    code = ("from dense_gemm_04_gb300 import phx\n"
            "print(phx.device_tag())\n"
            "print(phx.get_config(0, 3000, 3000, 3000))\n")
    first = _fresh_process(code, {})
    tag = first.stdout.splitlines()[0]
    p.write_text(f"{tag} 0 3000 3000 3000 TILE_M=64 TILE_N=128 TILE_K=8 STAGES=4\n")
    r = _fresh_process(code, {"PHX_TUNE_CACHE": str(p)})
    assert r.returncode == 0, r.stderr
    assert r.stdout.splitlines()[1] == "TILE_M=64 TILE_N=128 TILE_K=8 STAGES=4 FMA2=0", r.stdout


def test_no_multicast_configurations():
    # every f16 configuration is one CTA per 128-row tile or a 2-SM pair (TILE_M = 256); no
    # CLUSTER key is accepted (CTA pairs that multicast a B tile are not built)
    names = phx.config_names(phx.VARIANT_F16TC)
    assert not [n for n in names if "CLUSTER" in n], names
    for n in names:
        if n != "SKINNY":
            assert n.split()[0] in ("TILE_M=128", "TILE_M=256"), n
    for bad in ("TILE_M=256 TILE_N=256 TILE_K=64 STAGES=6 CLUSTER=2",
                "TILE_M=128 TILE_N=256 TILE_K=64 STAGES=4 CLUSTER=1"):
        with pytest.raises(phx.PhxError):
            phx.set_config(phx.VARIANT_F16TC, bad)
    with pytest.raises(phx.PhxError):
        phx.set_config(phx.VARIANT_SGEMM, "TILE_M=128 TILE_N=128 TILE_K=16 CLUSTER=2")
    phx.set_config(phx.VARIANT_F16TC, None)


def test_no_multicast_load_in_the_sources():
    # a TMA load with cluster multicast is not used anywhere in the library
    import pathlib
    csrc = pathlib.Path(__file__).resolve().parents[1] / "dense_gemm_04_gb300" / "csrc"
    for f in sorted(csrc.iterdir()):
        if f.suffix in (".cu", ".cuh", ".h", ".inc"):
            for i, line in enumerate(f.read_text().splitlines(), 1):
                assert not ("cp.async.bulk" in line and "multicast" in line), f"{f.name}:{i}: {line}"


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
