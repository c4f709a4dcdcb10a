"""Shared helpers of the parity tests: oracle-side expert records and the tolerance."""
import numpy as np

import synth
from oracle.formats import encode_record
from oracle.moe import RecordSource

REL_L2 = 5e-3          # ||y - y_ref|| / ||y_ref||
MAX_ABS_RMS = 2e-2     # max |y - y_ref| / rms(y_ref)


def oracle_experts(seed, H, I, fmt="nvfp4", scale=1.0):
    """Oracle RecordSource: weights regenerated on the CPU (times `scale`), quantised by
    the oracle in format fmt."""
    return RecordSource(
        lambda f: encode_record(*[w.numpy() * np.float32(scale)
                                  for w in synth.expert_weights(seed, f, H, I, "cpu")], fmt),
        H, I, fmt)


def oracle_shared(seed, layer, H, I, fmt="nvfp4"):
    from oracle.formats import decode_record
    rec = encode_record(*[w.numpy() for w in synth.shared_weights(seed, layer, H, I, "cpu")], fmt)
    return decode_record(rec, H, I, fmt)


def assert_close(y, y_ref, what=""):
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    nref = np.linalg.norm(y_ref)
    if nref == 0:
        assert np.all(y == 0), what
        return
    rel = np.linalg.norm(y - y_ref) / nref
    rms = nref / np.sqrt(y_ref.size)
    mx = np.max(np.abs(y - y_ref))
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e}"
    assert mx <= MAX_ABS_RMS * rms, f"{what}: max abs {mx:.3e} vs rms {rms:.3e}"
