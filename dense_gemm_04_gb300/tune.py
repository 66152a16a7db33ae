"""Command-line tuner: runs phx_autotune for one shape and prints its record.

    python -m dense_gemm_04_gb300.tune --shape 4096 4096 4096 [--variant sgemm|f16tc|both]
                                       [--save PATH]

For each variant it prints the configuration the library would launch untuned, the tuner's
record (every finalist with its median time and the SM clock sampled while it ran) and whether
the tuner's pick equals that default.  --save writes the tuning cache (keyed by device) to
PATH, which a later process loads with PHX_TUNE_CACHE=PATH.
"""
import argparse
import sys

from . import phx

_VARIANTS = {"sgemm": phx.VARIANT_SGEMM, "f16tc": phx.VARIANT_F16TC}


def main(argv=None) -> int:
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--shape", type=int, nargs=3, metavar=("M", "N", "K"), default=[4096, 4096, 4096])
    p.add_argument("--variant", choices=["sgemm", "f16tc", "both"], default="both")
    p.add_argument("--finalists", type=int, default=4)
    p.add_argument("--rounds", type=int, default=9)
    p.add_argument("--settle-ms", type=int, default=500)
    p.add_argument("--save", default=None)
    a = p.parse_args(argv)
    M, N, K = a.shape
    names = ["sgemm", "f16tc"] if a.variant == "both" else [a.variant]
    print(f"device {phx.device_tag()} shape {M} {N} {K}")
    for name in names:
        v = _VARIANTS[name]
        phx.set_config(v, None)
        default = phx.get_config(v, M, N, K)
        picked = phx.autotune(v, M, N, K, finalists=a.finalists, rounds=a.rounds, settle_ms=a.settle_ms)
        print(f"{name}: default {default}")
        print(phx.autotune_report(v).rstrip())
        print(f"{name}: picked == default: {picked == default}")
    if a.save:
        phx.tune_cache_save(a.save)
        print(f"tuning cache written to {a.save}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
