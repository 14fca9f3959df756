"""Shared helpers of the GPU tests: move a workload to the GPU, compare with the oracle."""
import numpy as np
import torch

MAX_ABS = 2e-2    # tolerance for bf16 inputs with fp32 accumulation, against the fp64 oracle
MEAN_ABS = 2e-3


def to_device(wl, device="cuda"):
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).view(dt).to(device)
    return dict(q=t(wl.q.view(np.int16), torch.bfloat16),
                k=t(wl.k.view(np.int16), torch.bfloat16),
                v=t(wl.v.view(np.int16), torch.bfloat16),
                user_offsets=t(wl.user_offsets, torch.int32),
                cand_to_user=t(wl.cand_to_user, torch.int32))


def out_f64(out, cands=None):
    x = out if cands is None else out[torch.as_tensor(cands, device=out.device)]
    return x.float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, what=""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max-abs {mx:.3e} mean-abs {mean:.3e}"
    return mx, mean
