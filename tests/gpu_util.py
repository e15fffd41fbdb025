"""Helpers shared by the GPU parity tests (device transfer and tolerances)."""
import numpy as np
import torch

from near_ties import NEAR_TIE  # noqa: F401  (rows below this oracle top-2 gap are counted, not failed)

# GEMM agreement with the float64 oracle (fp32 accumulation in any order).
REL_FRO = 1e-3
MAX_ABS_OVER_RMS = 1e-2


def dev():
    return torch.device("cuda:0")


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev()).view(torch.bfloat16)


def to_dev_i32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev())


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def packed_to_numpy(pk) -> dict:
    torch.cuda.synchronize()
    return dict(p0=pk.p0.cpu().numpy(), p1=pk.p1.cpu().numpy(), p2=pk.p2.cpu().numpy(),
                ebase=pk.ebase.cpu().numpy(), exc_off=pk.exc_off.cpu().numpy().view(np.uint32),
                exc_ent=pk.exc_ent.cpu().numpy().view(np.uint32)[:pk.n_exc], n_exc=pk.n_exc)


def assert_gemm_close(Y: np.ndarray, Y64: np.ndarray, what=""):
    Y = np.asarray(Y, dtype=np.float64)
    err = Y - Y64
    rel = np.linalg.norm(err) / max(np.linalg.norm(Y64), 1e-300)
    rms = np.sqrt(np.mean(Y64 ** 2))
    mx = np.abs(err).max()
    assert rel <= REL_FRO, f"{what}: rel Frobenius {rel:.3e}"
    assert mx <= MAX_ABS_OVER_RMS * rms, f"{what}: max abs {mx:.3e} vs rms {rms:.3e}"
    return rel, mx / rms


def new_status():
    return torch.zeros(1, dtype=torch.int32, device=dev())


def status_value(st):
    torch.cuda.synchronize()
    return int(st.item())


# Tree attention vs the float64 oracle: P rounded to bf16 for the P.V product
# (relative error <= 2^-9 per weight) and O rounded to bf16 (<= 2^-9 of the
# element): about 1.6e-3 rms relative in all. Per element the error is bounded
# by a small fraction of the output's rms (the P rounding, spread over many
# keys) plus 2^-8 of the element itself (the O rounding, and the P rounding in
# rows with few keys, where |O| can reach max |V|, far above the rms).
ATTN_REL_FRO = 4e-3
ATTN_MAX_ABS_OVER_RMS = 3e-2
ATTN_ELEM_REL = 2.0 ** -8


def assert_attn_close(O_bits: np.ndarray, O64: np.ndarray, what=""):
    O = (O_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    err = O - O64
    rel = np.linalg.norm(err) / max(np.linalg.norm(O64), 1e-300)
    rms = np.sqrt(np.mean(O64 ** 2))
    bound = ATTN_MAX_ABS_OVER_RMS * rms + ATTN_ELEM_REL * np.abs(O64)
    mx = np.abs(err).max()
    assert np.isfinite(O).all(), f"{what}: non-finite output"
    assert rel <= ATTN_REL_FRO, f"{what}: rel Frobenius {rel:.3e}"
    worst = np.unravel_index(np.argmax(np.abs(err) - bound), err.shape)
    assert (np.abs(err) <= bound).all(), \
        f"{what}: |err| {abs(err[worst]):.3e} at {worst} (O {O64[worst]:.4f}) above {bound[worst]:.3e} (rms {rms:.3e})"
    return rel, mx / rms
