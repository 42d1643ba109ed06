"""The debug build (block_sparse_attention_token_gb300.build.build(debug=True),
loaded when SPARSP_DEBUG=1): the same kernels with every address they derive
themselves - TMA coordinates, output rows, list and CSR write positions -
checked, reporting SPARSP_ERR_DATA instead of an out-of-range access. On the
small workloads (every block size and head dimension, odd block counts, both
dtypes) none of the checks may fire and the results must match the oracle.
It runs in a child process so that this process keeps the release library."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.timeout(1500)]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r})
    import numpy as np
    import torch
    import block_sparse_attention_token_gb300 as sp
    assert sp.DEBUG and sp.LIB_PATH.endswith("libsparsp_debug.so")
    import synth
    from oracle import sparsp_oracle as orc
    from tests.gpu_helpers import OracleChain, compare_csr, compare_values, dev, host, status_word
    from tests.test_gpu_steps import SMALL
    for name in ["tiny", "medium", "r128", "r64", "r64odd", "r128d64", "wave"]:
        wl = SMALL[name]
        data = synth.make(wl)
        shape = sp.shape_of(wl)
        ch = OracleChain(wl, data)
        st = status_word()
        rp, ci = sp.select(shape, torch.from_numpy(ch.S32).cuda(), wl.top_p, wl.k_floor, status=st)
        q, k, v = (dev(x, wl) for x in (ch.qb, ch.kb, ch.vb))
        dem = sp.kv_demand(shape, wl.P, rp, ci, k, v, status=st)
        o, lse = sp.attn_fwd(shape, q, k, v, rp, ci, status=st)
        grads = None
        if wl.dtype == "bf16":
            do = synth.round_bf16(np.random.default_rng(wl.seed + 300).standard_normal(data["q"].shape,
                                                                                      dtype=np.float32))
            dob = orc.reorder(do, ch.g)
            grads = sp.attn_bwd(shape, q, k, v, o, lse, dev(dob, wl), rp, ci, status=st)
        pipe = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, backward=False)
        kw = {{}}
        if wl.estimator == "lowrank":
            kw = dict(wq=torch.from_numpy(data["wq"]).cuda(), wk=torch.from_numpy(data["wk"]).cuda())
        pipe.forward(*(dev(data[x], wl) for x in ("q", "k", "v")), **kw)
        torch.cuda.synchronize()
        assert st.item() == 0 and pipe.status.item() == 0, (name, st.item(), pipe.status.item())
        assert compare_csr(host(rp), host(ci), ch.sel) == 0, name
        ref = orc.kv_demand(ch.sel.row_ptr, ch.sel.col_idx, ch.g.B, ch.g.H, ch.g.nb, wl.P, ch.g.Bt, ch.g.d,
                            wl.elem_bytes)
        assert np.array_equal(host(dem.dem_idx)[:int(ref.dem_ptr[-1])], ref.dem_idx), name
        O, L = orc.attn_fwd(ch.qb, ch.kb, ch.vb, ch.sel.row_ptr, ch.sel.col_idx, ch.g.Bt, ch.scale)
        compare_values(host(o), O, wl, name + " O")
        compare_values(host(lse), L, wl, name + " LSE")
        if grads is not None:
            dQ, dK, dV = orc.attn_bwd(ch.qb, ch.kb, ch.vb, dob, ch.sel.row_ptr, ch.sel.col_idx, ch.g.Bt, ch.scale)
            for got, want, what in zip(grads, (dQ, dK, dV), ("dQ", "dK", "dV")):
                compare_values(host(got), want, wl, name + " " + what)
        print(name, "clean")
    print("debug build OK")
""")


def test_debug_build_runs_clean():
    from block_sparse_attention_token_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, SPARSP_DEBUG="1")
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT)], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=1400)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "debug build OK" in r.stdout
