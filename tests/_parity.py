"""GPU-vs-oracle comparison helpers (tolerances of the decode contract:
out max |err| <= 2e-2 and per-row cosine >= 0.9999 against the fp64 oracle,
|delta lse| <= 1e-3, row selection bit-exact)."""
import numpy as np
import torch

import oracle
from swa_paged_decode_gb300 import binding as B
from swa_paged_decode_gb300 import workloads as W

OUT_ATOL = 2e-2
COS_MIN = 0.9999
LSE_ATOL = 1e-3


def oracle_ref(w: W.Workload, tokens=None):
    a = W.oracle_args(w)
    return oracle.decode(a["q"], a["caches"], a["lists"], scale=a["scale"], sink=a["sink"],
                         positions=a["positions"], cos_sin=a["cos_sin"], rope_style=a["rope_style"], tokens=tokens)


def run_gpu(w: W.Workload, num_sms: int = 0):
    dec = B.Decoder(w, num_sms=num_sms)
    out, lse = dec(w)
    kept, chk = dec.selection()
    torch.cuda.synchronize()
    assert B.dsa_decode_read_status(dec.workspace) == 0
    return dec, out, lse, kept, chk


def compare(out, lse, kept, chk, ref, tokens=None, what="", out_scale=1.0):
    """GPU result vs oracle. ``out_scale``: the absolute bound on out is
    applied to out * out_scale (for KV rows drawn at 2^k times unit scale, a
    scale of 2^-k puts the output back on the unit scale the bound is
    stated for); the cosine, lse and selection checks do not depend on it."""
    r_out, r_lse, r_kept, r_chk = ref
    if tokens is None:
        tokens = np.arange(out.shape[0])
    tok = torch.as_tensor(np.asarray(tokens), device=out.device, dtype=torch.long)
    o = out.index_select(0, tok).float().cpu().double().numpy()
    l = lse.index_select(0, tok).cpu().double().numpy()
    k = kept.index_select(0, tok).cpu().numpy()
    c = chk.index_select(0, tok).cpu().numpy().view(np.uint32)
    # row selection: bit exact
    assert np.array_equal(k, r_kept), f"{what}: kept rows differ"
    assert np.array_equal(c, r_chk), f"{what}: selection checksum differs"
    # lse
    fin = np.isfinite(r_lse)
    assert np.array_equal(np.isfinite(l), fin), f"{what}: -inf pattern of lse differs"
    assert np.all(l[~fin] == r_lse[~fin])
    if fin.any():
        dl = np.abs(l[fin] - r_lse[fin]).max()
        assert dl <= LSE_ATOL, f"{what}: max |dlse| = {dl}"
    # out
    err = np.abs(o - r_out).max() * out_scale if o.size else 0.0
    assert err <= OUT_ATOL, f"{what}: max |err| = {err}"
    rn = np.linalg.norm(r_out, axis=-1)
    zero = rn == 0
    assert np.all(o[zero] == 0), f"{what}: rows that must be zero are not"
    on = np.linalg.norm(o, axis=-1)
    nz = ~zero
    if nz.any():
        cos = (o * r_out).sum(-1)[nz] / (on[nz] * rn[nz])
        assert cos.min() >= COS_MIN, f"{what}: min cosine = {cos.min()}"
    return dict(max_err=float(err), max_dlse=float(np.abs(l[fin] - r_lse[fin]).max()) if fin.any() else 0.0)
