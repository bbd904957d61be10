"""The five verification workloads end to end (plan -> verify every layer ->
accept -> commit -> one readback -> pool release), step by step against the
oracle: integers bit-exact for every request; FP32 states and bf16 outputs
within tolerance for the requests followed in FP64."""
import pytest
import torch

import gdnsynth as sy
from gpu_util import build_lib
from workload_harness import Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_dev):
    build_lib()


def test_tiny_workload(cuda_dev):
    w = Workload(sy.SPECS["tiny"], 1, [0], cuda_dev)
    res = w.step(0)
    assert res.accept_len[0] == 2          # drafts match for the first two rows, miss on the third
    w.check_states()


def test_batch1_workload(cuda_dev):
    w = Workload(sy.SPECS["batch1"], 3, [0], cuda_dev)
    for s in range(3):
        w.step(s)
        w.check_states()


def test_continuous_batch_16x30_layers_200_steps(cuda_dev):
    spec = sy.SPECS["cb16"]
    w = Workload(spec, spec.steps, [0, 5, 10, 15], cuda_dev)
    for s in range(spec.steps):
        w.step(s)
        if s in (0, 1, 50, 100, spec.steps - 1):
            w.check_states()
    st = w.vs.stats.cpu().tolist()
    assert st[4] == spec.steps


def test_paged_256_requests_full_size(cuda_dev):
    spec = sy.SPECS["paged256"]
    free, total = torch.cuda.mem_get_info()
    if free < 130 * 2 ** 30:
        pytest.fail("needs ~125 GB of free device memory, found %.1f GB" % (free / 2 ** 30))
    w = Workload(spec, 4, [0, 1, 16, 100, 150, 200, 254, 255], cuda_dev, gen_device=cuda_dev)
    for s in range(4):
        w.step(s)
        w.check_states()
    # the 16 requests that shared a prefix slot moved to fresh slots at the first commit
    assert len(set(w.slots_m[:16])) == 16 and w.slot_of0[0] not in w.slots_m
