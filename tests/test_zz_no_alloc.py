"""moe_expert_ffn_noalloc: the decode expert FFN for callers that cannot
allocate device memory - an engine whose device memory an outer framework
reserved up front, a serving loop that must not block on the allocator, a
plugin handed only its buffers.  Its scratch is a fixed array inside the
library.  Through the C ABI, two calls in a row must give the same layer
output as the workspace-taking moe_expert_ffn on the same inputs, within the
output tolerance the other parity tests use, without changing the device's
free memory; sizes beyond the array are refused.  Collected last on
purpose."""
import numpy as np
import pytest
import torch

import gen
from tests.helpers import TOL

pytestmark = pytest.mark.gpu


def _buffers(T, H, E, k):
    i32, f32 = torch.int32, torch.float32
    return {n: torch.zeros(sz, dtype=dt, device="cuda") for n, sz, dt in (
        ("ids", T * k, i32), ("w", T * k, f32), ("p", T * k, f32), ("lg", T * E, f32),
        ("counts", E, i32), ("off", E + 1, i32), ("perm", T * k, i32), ("inv", T * k, i32),
        ("src", E, i32), ("act", E, i32), ("nact", 2, i32), ("miss", E, i32), ("nmiss", 1, i32),
        ("st", 1, i32))}


def _prepare(moe, dw, z, xd, T, s):
    wl = dw.wl
    ra = moe.moe_route_args()
    ra.x, ra.w_router, ra.bias = xd.data_ptr(), dw.w_router[0].data_ptr(), None
    ra.T, ra.H, ra.E, ra.k = T, wl.H, wl.E, wl.k
    ra.ids, ra.w, ra.p_sel, ra.logits = (z[n].data_ptr() for n in ("ids", "w", "p", "lg"))
    moe.moe_route(ra, s)
    moe.moe_permute(z["ids"].data_ptr(), T, wl.k, wl.E, z["counts"].data_ptr(),
                    z["off"].data_ptr(), z["perm"].data_ptr(), z["inv"].data_ptr(), 0, 128,
                    z["st"].data_ptr(), s)
    moe.expcache_lookup(dw.cache.handle, 0, z["counts"].data_ptr(), z["src"].data_ptr(),
                        z["act"].data_ptr(), z["nact"].data_ptr(), z["miss"].data_ptr(),
                        z["nmiss"].data_ptr(), z["st"].data_ptr(), s)


def _args(moe, dw, z, xd, T, o, os_, Is):
    wl = dw.wl
    fa = moe.moe_ffn_args()
    fa.mode, fa.stages, fa.T, fa.H, fa.I, fa.E, fa.k = 0, 3, T, wl.H, wl.I, wl.E, wl.k
    fa.x, fa.cache, fa.gscale = xd.data_ptr(), dw.cache.handle, dw.gscale[0].data_ptr()
    fa.src_slot, fa.act_list, fa.n_act = (z[n].data_ptr() for n in ("src", "act", "nact"))
    fa.offsets, fa.perm, fa.w = z["off"].data_ptr(), z["perm"].data_ptr(), z["w"].data_ptr()
    fa.group, fa.n_stage, fa.Is = 0, 0, Is
    if Is:
        fa.s_gate, fa.s_up, fa.s_down = (t.data_ptr() for t in dw.shared[0])
    fa.o_route, fa.o_shared = o.data_ptr(), (os_.data_ptr() if Is else None)
    fa.status = z["st"].data_ptr()
    return fa


def _layer_out(o, os_, inv, T, k, H):
    o = o.double().view(T * k, H).cpu().numpy()
    inv = inv.cpu().numpy()[:T * k]
    y = np.stack([o[inv[t * k:(t + 1) * k]].sum(0) for t in range(T)])
    return y if os_ is None else y + os_.double().view(T, H).cpu().numpy()


def _max_tokens(I, k, Is, limit):
    """Largest T whose decode scratch (T*k*I + T*Is floats + 256 bytes) fits."""
    return (limit - 256) // ((k * I + Is) * 4)


# (tokens, shared expert on): one and two tokens, and the largest T the
# fixed scratch holds for the 6144 x 2048 top-8 layer with and without the
# shared expert (113 and 127)
@pytest.mark.parametrize("T,shared", [(1, True), (2, True), (113, True), (127, False)])
def test_noalloc_entry_point_matches_workspace_entry_point(T, shared):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import gen.device as gd
    from routed_expert_layer_router_gb300 import moe
    wl = gen.WORKLOADS["decode"]
    H, I, E, k = wl.H, wl.I, wl.E, wl.k
    Is = wl.Is if shared else 0
    T_fit = _max_tokens(I, k, Is, moe.MOE_NOALLOC_SCRATCH_BYTES)
    assert T <= T_fit
    dw = gd.build(wl, T_max=T + 1)
    try:
        s = torch.cuda.current_stream().cuda_stream
        z = _buffers(T + 1, H, E, k)
        ws_b = moe.moe_ffn_workspace_bytes(0, T, H, I, E, k, Is)
        ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
        for call, draw in enumerate((10, 20)):  # two calls in a row
            xd = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
            gen.dev_x_bf16(wl.seed, 0, draw, T, H, xd.data_ptr(), s)
            _prepare(moe, dw, z, xd, T, s)
            o_ref = torch.zeros((T * k, H), dtype=torch.float32, device="cuda")
            os_ref = torch.zeros((T, H), dtype=torch.float32, device="cuda")
            fa = _args(moe, dw, z, xd, T, o_ref, os_ref, Is)
            fa.workspace, fa.workspace_bytes = ws.data_ptr(), ws_b
            moe.moe_expert_ffn(fa, s)
            o_na = torch.full((T * k, H), float("nan"), dtype=torch.float32, device="cuda")
            os_na = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
            fb = _args(moe, dw, z, xd, T, o_na, os_na, Is)
            fb.workspace, fb.workspace_bytes = None, 0
            torch.cuda.synchronize()
            free0 = torch.cuda.mem_get_info()[0]
            moe.moe_expert_ffn_noalloc(fb, s)
            torch.cuda.synchronize()
            assert torch.cuda.mem_get_info()[0] == free0, f"call {call}: device memory changed"
            assert z["st"].item() == 0
            y_ref = _layer_out(o_ref, os_ref if shared else None, z["inv"], T, k, H)
            y_na = _layer_out(o_na, os_na if shared else None, z["inv"], T, k, H)
            rms = np.sqrt(np.mean(y_ref ** 2))
            assert np.isfinite(y_na).all(), f"call {call}"
            assert np.abs(y_na - y_ref).max() <= TOL * rms, f"call {call}"
        # one token more than the fixed scratch holds, and a prefill-sized
        # chunk, are refused before any work is queued
        for T_big in (T_fit + 1, 4096):
            big = _args(moe, dw, z, xd, T_big, o_na, os_na, Is)
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_expert_ffn_noalloc(big, s)
            assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
    finally:
        dw.close()
