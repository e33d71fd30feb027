"""Small, self-checking invocations of one layer variant each, sized for
profiler captures (a few GB on the device at most, three calls):

    python -m mixture_experts_ffn_softmax_gb300.profile_cases <case> [auto|single|pairs]

Cases:
  fp8_mixtral_m2048     FP8 W8A8 layer, Mixtral-8x7B expert shape, M = 2048
  fp8block_mixtral_m2048  the same with 128 x 128 weight-block scales
  int4_mixtral_decode   int4 (group 128, zero points) layer, Mixtral shape, M = 16
  mxfp4_mixtral_decode  MX FP4 layer, Mixtral shape, M = 16
  int4_mixtral_m2048    int4 (group 128) layer, Mixtral shape, M = 2048
The optional second argument picks the GEMM tile mode (default auto).
Exits non-zero if the layer reports an error."""
import dataclasses
import sys

import torch

from . import workloads as wl
from . import (alloc_workspace, moe_forward_fp8, moe_forward_wq, moe_route, read_error,
               set_gemm_tiles, workspace_error_word, workspace_size, workspace_size_fp8)


def _spec(M):
    return dataclasses.replace(wl.SPECS["mixtral_prefill"], M=M, name=f"mixtral_m{M}")


def run(case: str, calls: int = 3, tiles: str = "auto") -> None:
    set_gemm_tiles(tiles)
    kind, _, shape = case.partition("_mixtral_")
    M = 16 if shape == "decode" else int(shape.lstrip("m"))
    spec = _spec(M)
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    w, ids = moe_route(d["router_logits"], spec.top_k, "softmax", True)
    out = torch.empty_like(d["hidden"])
    if kind in ("fp8", "fp8block"):
        q = wl.make_fp8_weights(spec, device="cuda", block=kind == "fp8block")
        ws = alloc_workspace(workspace_size_fp8(spec.M, spec.H, spec.I, spec.E, spec.top_k))
        for _ in range(calls):
            moe_forward_fp8(d["hidden"], w, ids, q["w13_q"], q["w2_q"], q["w13_scale"],
                            q["w2_scale"], workspace=ws, out=out)
    else:
        q = wl.make_wq_weights(spec, kind, 128 if kind == "int4" else 32, device="cuda")
        ws = alloc_workspace(workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k,
                                            "separate"))
        for _ in range(calls):
            moe_forward_wq(d["hidden"], w, ids, kind, q["w13_q"], q["w2_q"], q["w13_scale"],
                           q["w2_scale"], q["w13_zero"], q["w2_zero"], q["group_size"],
                           workspace=ws, out=out)
    torch.cuda.synchronize()
    err = read_error(workspace_error_word(ws))
    if err != 0 or not torch.isfinite(out.float()).all():
        raise SystemExit(f"{case}: error word {err}")
    print(f"{case}: ok")


if __name__ == "__main__":
    run(sys.argv[1], tiles=sys.argv[2] if len(sys.argv) > 2 else "auto")
