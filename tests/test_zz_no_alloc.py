"""ep_get_layout_static_scratch: the layout entry point for callers that cannot allocate
device memory (its workspace is a fixed array inside libep.so instead of a buffer the
caller hands over). Checked through the C ABI against ep_get_layout, which takes a
caller-allocated workspace: two calls in a row (different routing each time, so the
second call runs over the first call's leftovers in the shared array) must give
bit-identical outputs. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _outputs(lb):
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in lb.as_dict().items()}


def test_static_scratch_layout_matches_workspace_layout_twice():
    from combine_layout_02_gb300 import build
    build.build()
    import combine_layout_02_gb300 as ep
    from combine_layout_02_gb300.buffers import LayoutBuffers
    import workloads

    L = ep.lib()
    w = workloads.CONFIGS["dsv3"]
    for call, seed in enumerate((11, 12)):
        wl = workloads.Workload("nl", R=w.R, T=w.T, H=w.H, E=w.E, k=w.k, C=w.C, seed=seed)
        topk = torch.from_numpy(workloads.make_workload(wl, with_hidden=False)["topk_idx"]).cuda()
        sh = ep.make_shape(wl.R, wl.T, wl.H, wl.E, wl.k, wl.C)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        launch = ep.make_launch(error_flags=err)

        ref = LayoutBuffers(sh)
        st = L.ep_get_layout(ctypes.byref(sh), ctypes.c_void_p(topk.data_ptr()),
                             ctypes.byref(ref.layout()), ctypes.byref(ref.handle()),
                             ctypes.c_void_p(ref.workspace.data_ptr()),
                             ref.workspace.numel(), ctypes.byref(launch))
        assert st == ep.EP_OK
        got = LayoutBuffers(sh)
        for t in got.as_dict().values():
            t.fill_(0x5A if t.dtype == torch.uint8 else -77)
        st = L.ep_get_layout_static_scratch(ctypes.byref(sh), ctypes.c_void_p(topk.data_ptr()),
                                            ctypes.byref(got.layout()), ctypes.byref(got.handle()),
                                            ctypes.byref(launch))
        assert st == ep.EP_OK, f"call {call}: status {st}"
        a, b = _outputs(ref), _outputs(got)
        for key in a:
            np.testing.assert_array_equal(b[key], a[key], err_msg=f"call {call}: {key}")
        assert int(err.item()) == 0


def test_static_scratch_rejects_shapes_beyond_its_size():
    import combine_layout_02_gb300 as ep
    L = ep.lib()
    # R=64, C=64, E=8192 needs 64*64*64*4 + 64*64*8192*4 bytes of scratch (> 256 KiB)
    sh = ep.make_shape(64, 256, 128, 8192, 8, C=64)
    assert L.ep_layout_workspace_size(ctypes.byref(sh)) > 256 * 1024
    h = ep.ep_handle(0x1000, 0x1000, 0x1000, None, 0x1000, 0x1000, 0x1000)
    launch = ep.make_launch()
    st = L.ep_get_layout_static_scratch(ctypes.byref(sh), ctypes.c_void_p(0x2000), None,
                                        ctypes.byref(h), ctypes.byref(launch))
    assert st == ep.EP_ERR_UNSUPPORTED
