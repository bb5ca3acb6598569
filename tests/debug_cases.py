"""One small case for every kernel of the library, run through whichever
libmuon the process loads (MUON_LIB_PATH selects the -DMUON_DEBUG build).

    python tests/debug_cases.py OUT.npz

Saves every result array and every call's muon_query_status code to OUT.npz.
tests/test_gpu_debug_build.py runs it under the release and the debug
library and compares the two files: same bits, and no status code set.
"""
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
from newton_schulz_gb300 import binding, synth  # noqa: E402

HP = dict(mu=0.95, nesterov=True, lr=0.02, wd=0.01, scale_rule=0)
ENV_KEYS = ("MUON_GEMM_PAIR", "MUON_GEMM_WIDE", "MUON_MAX_KSPLIT", "MUON_GRAM_SPACE",
            "MUON_SMALL_PATH")


def _env(**kw):
    for k in ENV_KEYS:
        os.environ.pop(k, None)
    for k, v in kw.items():
        os.environ[k] = v


def main(out_path):
    binding.load()
    res, codes = {}, {}

    def step(name, groups, **env):
        _env(**env)
        binding.muon_step_grouped(groups, **HP)
        torch.cuda.synchronize()
        codes[name] = binding.muon_query_status()
        for i, g in enumerate(groups):
            res[f"{name}.W{i}"] = g["W"].float().cpu().numpy()
            res[f"{name}.M{i}"] = g["Mom"].cpu().numpy()

    def ns(name, shape, seed, cfg=None, **env):
        _env(**env)
        x = torch.randn(shape, generator=torch.Generator().manual_seed(seed)).cuda()
        out = torch.empty_like(x)
        binding.muon_ns_batched_ex(x, cfg or binding.make_config(), out)
        torch.cuda.synchronize()
        codes[name] = binding.muon_query_status()
        res[name] = out.cpu().numpy()

    # fused small-m kernel: fp32 and bf16 weights, both layouts
    step("small_c1", synth.config_c1("cuda"))
    step("small_bf16w", [synth.random_group((3, 512, 48), torch.bfloat16, torch.bfloat16, "cuda", 1, 1e-3),
                         synth.random_group((2, 40, 1000), torch.float32, torch.float32, "cuda", 2, 1.0, 0.5)])
    # grouped GEMM path: ragged shapes, both layouts, bf16 weights
    step("gemm_mixed", [synth.random_group((2, 200, 333), torch.float32, torch.float32, "cuda", 3, 1.0),
                        synth.random_group((1, 520, 300), torch.bfloat16, torch.bfloat16, "cuda", 4, 1e-3)])
    # split-K Gram (tall-skinny), the generic path for a small shape
    ns("splitk", (1, 96, 10240), 5)
    ns("generic_small", (2, 24, 2048), 6, MUON_SMALL_PATH="0")
    # CTA pairs forced, with and without split-K
    ns("pairs", (2, 640, 2048), 7, MUON_GEMM_PAIR="1", MUON_GEMM_WIDE="0", MUON_MAX_KSPLIT="1")
    # WIDE blocks forced (an odd number of row tiles: an empty second half)
    ns("wide", (2, 640, 1000), 13, MUON_GEMM_WIDE="1", MUON_MAX_KSPLIT="1")
    # high-precision mode on both paths
    ns("precise_gemm", (1, 300, 700), 8, binding.make_config(precision=binding.NS_TF32))
    ns("precise_small", (2, 48, 900), 9, binding.make_config(precision=binding.NS_TF32))
    # Gram space, forced, with a restart
    ns("gram_space", (1, 256, 1024), 10, MUON_GRAM_SPACE="force")
    # allocation-free entry point
    _env()
    x = torch.randn((2, 256, 512), generator=torch.Generator().manual_seed(11)).cuda().bfloat16()
    binding.muon_ns_batched_noalloc(x, 5, 3.4445, -4.7750, 2.0315)
    torch.cuda.synchronize()
    codes["noalloc"] = binding.muon_query_status()
    res["noalloc"] = x.float().cpu().numpy()
    # AdamW for non-matrix parameters
    g = torch.Generator().manual_seed(12)
    p = torch.randn(1000, generator=g).cuda()
    grad = torch.randn(1000, generator=g).cuda()
    m, v = torch.zeros_like(p), torch.zeros_like(p)
    binding.muon_adamw_grouped([dict(param=p, grad=grad, exp_avg=m, exp_avg_sq=v)], step=1,
                               lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    torch.cuda.synchronize()
    codes["adamw"] = binding.muon_query_status()
    res["adamw"] = p.cpu().numpy()

    np.savez(out_path, codes=np.array([codes[k] for k in sorted(codes)]),
             names=np.array(sorted(codes)), debug_build=np.array(binding.muon_debug_build()), **res)


if __name__ == "__main__":
    main(sys.argv[1])
