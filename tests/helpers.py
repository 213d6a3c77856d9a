"""Test plumbing: numpy arrays from the seeded generators -> torch CUDA
tensors for the library, and the parity bars.  No attention arithmetic."""
import numpy as np
import torch

# Parity bars (stated with the method): bf16 outputs |err| <= ATOL + RTOL*|ref|,
# lse |err| <= LSE_ATOL; page writes and INT8 codes bit-exact.
ATOL, RTOL, LSE_ATOL = 1e-2, 1e-2, 1e-3


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def host_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def check_out(out_gpu: torch.Tensor, ref: np.ndarray, what=""):
    got = host_f32(out_gpu).astype(np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = ~(err <= ATOL + RTOL * np.abs(ref))          # NaN counts as outside
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outputs outside "
                             f"{ATOL}+{RTOL}|ref|; first at {tuple(i)}: got "
                             f"{got[tuple(i)]}, ref {ref[tuple(i)]}, max err {np.nanmax(err):.3e}")


def check_lse(lse_gpu: torch.Tensor, ref: np.ndarray, what=""):
    got = lse_gpu.detach().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape
    both_inf = np.isneginf(got) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(got - ref))
    assert not np.isnan(err).any(), f"{what}: NaN in lse"
    assert err.max() <= LSE_ATOL, f"{what}: lse max err {err.max():.3e}"
