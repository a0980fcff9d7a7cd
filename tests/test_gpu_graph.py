"""Library calls captured into a CUDA graph and replayed give the eager bits.
(The workspace of the tensor-core dot is allocated before capture.)"""
import numpy as np
import pytest

import synth
from gpu_util import loom_module, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = require_gpu()
    return torch, loom_module()


def test_capture_and_replay(env):
    torch, loom = env
    s = torch.cuda.Stream()
    seg = synth.batched_segments(num_segments=3000)
    bat = synth.dequant_batched(n_rows=512, k=2048, batch=16, seed=3)
    pd = synth.packed_dot_case(problems=4, records=20, lanes=1024, streams=64, counts=[20, 3, 0, 17], seed=4)
    ls = synth.lane_segments(num_segments=300, rows=64, lanes=32, width=4, seed=5)
    rc = synth.routed_case(tokens=40, routes=8, width=512, seed=6)
    d = dict(v=to_dev(seg["values"], torch), c=to_dev(seg["counts"], torch), i=to_dev(seg["initial"], torch),
             w=to_dev(bat["w"].view("<i4"), torch), sw=to_dev(bat["scale_w"], torch),
             x=to_dev(bat["x"].view("<i4"), torch), sx=to_dev(bat["scale_x"], torch),
             pf=to_dev(pd["fields"], torch), ps=to_dev(pd["scales"].view(np.int16), torch), pr=to_dev(pd["rhs"], torch),
             pc=to_dev(pd["counts"], torch), pi=to_dev(pd["initial"], torch),
             lv=to_dev(ls["values"], torch), lc=to_dev(ls["counts"], torch),
             ri=to_dev(rc["ids"], torch), rw=to_dev(rc["weights"], torch), rp=to_dev(rc["payload"], torch))
    f32, i32 = torch.float32, torch.int32
    out = dict(seg=tuple(torch.empty(3000, dtype=t, device="cuda") for t in (i32, i32, f32, f32)),
               y=torch.empty((512, 16), dtype=f32, device="cuda"),
               pd=torch.empty((4, 1024), dtype=f32, device="cuda"),
               ls=torch.empty((300, 32), dtype=f32, device="cuda"),
               gr=torch.empty((300, 32), dtype=f32, device="cuda"),
               rc=torch.empty((40, 512), dtype=f32, device="cuda"))
    ws = loom.dot_workspace(512, 2048, 16)

    def calls():
        loom.loom_row_sum_batched(d["v"], 3000, 2016, 63, 32, d["c"], d["i"], 8, out=out["seg"], stream=s)
        loom.loom_i8_dequant_dot(d["w"], d["sw"], 512, 2048, d["x"], d["sx"], 16, y=out["y"], workspace=ws,
                                 stream=s)
        loom.loom_packed_dot(d["pf"], d["ps"], d["pr"], d["pc"], 0, d["pi"], out=out["pd"], stream=s)
        loom.loom_sum_rows(d["lv"], 300, 64 * 128, 64, 32, 4, d["lc"], 0, out=out["ls"], stream=s)
        loom.loom_sum_guarded_rows(d["lv"], 300, 64 * 128, 64, 32, d["lc"], 0, 3, 30, out=out["gr"], stream=s)
        loom.loom_routed_combine(d["ri"], d["rw"], d["rp"], out=out["rc"], stream=s)

    def snapshot():
        return [t.clone() for t in out["seg"]] + [out[k].clone() for k in ("y", "pd", "ls", "gr", "rc")]

    with torch.cuda.stream(s):
        calls()
    s.synchronize()
    eager = snapshot()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
    for t in list(out["seg"]) + [out[k] for k in ("y", "pd", "ls", "gr", "rc")]:
        t.fill_(-1)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(snapshot(), eager):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
