"""Device-side error reporting, exercised without faulting the GPU: a token id
outside the vocabulary and a bounded wait that runs out both set the
workspace error word; the context stays usable afterwards."""
import numpy as np
import pytest
import torch

import nc_synth
from pretraining_step_pretrain_b300 import build, nc
from tests.helpers import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    nc.lib()


def _step(ids, tg, w, shape=nc_synth.SMALL.shape):
    st = nc.Step(shape, "bf16", ids.shape[0], ids.shape[1], w)
    loss = st.run(torch.from_numpy(ids).cuda(), torch.from_numpy(tg).cuda())
    torch.cuda.synchronize()
    return st, float(loss.item())


def test_token_id_out_of_range_is_reported():
    ids, tg, w = inputs(nc_synth.SMALL.shape, 2, 64, "bf16")
    bad = ids.copy()
    bad[1, 7] = nc_synth.SMALL.shape.vocab + 5
    st, _ = _step(bad, tg, w)
    assert st.status() == 6                       # NC_ERR_TOKEN_RANGE
    assert st.status() == 0                       # reading clears the word
    st2, loss = _step(ids, tg, w)                 # the context still works
    assert st2.status() == 0 and np.isfinite(loss)


def test_target_out_of_range_is_reported():
    ids, tg, w = inputs(nc_synth.SMALL.shape, 2, 64, "bf16")
    bad = tg.copy()
    bad[0, 3] = -7
    st, _ = _step(ids, bad, w)
    assert st.status() == 6


def test_bounded_wait_times_out_with_status():
    ws = nc.alloc_workspace(1024, "cuda")
    nc.selftest_wait_timeout(2000, ws)            # 2 ms limit on a barrier nothing completes
    assert nc.get_device_status(ws) == 5          # NC_ERR_TIMEOUT
    assert nc.get_device_status(ws) == 0
    ids, tg, w = inputs(nc_synth.SMALL.shape, 2, 64, "bf16")
    st, loss = _step(ids, tg, w)
    assert st.status() == 0 and np.isfinite(loss)
