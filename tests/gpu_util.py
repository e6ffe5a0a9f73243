"""Helpers shared by the GPU tests: device copies of the seeded inputs and
the tolerance checks against the fp64 oracle."""
import numpy as np

# bf16 path (max |err| and relative Frobenius error); fp32 path (max |err|)
BF16_MAX_ABS = 2e-2
BF16_REL_FRO = 5e-3
F32_MAX_ABS = 1e-4


def to_dev_bf16(bits, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def to_dev_i32(a, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def to_host_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite output"
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / den if den > 0 else float(np.linalg.norm(got - ref))
    return err, rel


def assert_bf16_close(got, ref, what=""):
    err, rel = errors(got, ref)
    assert err <= BF16_MAX_ABS and rel <= BF16_REL_FRO, \
        f"{what}: max|err|={err:.3g} (<= {BF16_MAX_ABS}), rel_fro={rel:.3g} (<= {BF16_REL_FRO})"
    return err, rel


def assert_f32_close(got, ref, what=""):
    err, _ = errors(got, ref)
    assert err <= F32_MAX_ABS, f"{what}: max|err|={err:.3g} (<= {F32_MAX_ABS})"
    return err
