"""The bounded waits of the attention kernels, made to run out on purpose without any fault: the
test entry point zf_decode_attn_wait_test shortens the limit of the waits for the metadata warp's
items and delays that warp's first item beyond it.  The call must report ZF_DEV_TIMEOUT in the
status word and return; the context and the stream stay usable, and the next ordinary call on the
same stream is correct against the float64 oracle."""
import pytest
import torch

from decode_attention_compressed_gb300 import inputs as I
from oracle import zf_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zf():
    return H.zf_module()


@pytest.mark.parametrize("kernel", ["warp_mma", "tcgen05"])
def test_a_wait_that_runs_out_reports_timeout_and_the_next_call_is_correct(zf, kernel):
    w = I.Workload("case", 3, 14, 2, 16, 300, pool="random", seed=5)
    layer = I.make_layer(w, seq_lens=[300, 48, 1])
    gc = H.gpu_cache_from(layer, zf)
    dev = torch.device("cuda")
    q, table, lens = layer.q.to(dev), layer.page_table.to(dev), layer.seq_lens.to(dev)
    # 200 us limit, first item 20 ms late: every wait for it runs out
    zf.decode_attn_wait_test(gc, q, table, lens, layer.scale, kernel=kernel, wait_limit_ns=200_000,
                             publish_delay_ns=20_000_000)
    torch.cuda.synchronize()
    assert gc.status_word() & zf.DEV_TIMEOUT
    gc.status.zero_()
    # the same entry point with the delay under the limit finishes normally
    o1, l1 = zf.decode_attn_wait_test(gc, q, table, lens, layer.scale, kernel=kernel, wait_limit_ns=500_000_000,
                                      publish_delay_ns=1_000_000)
    out, lse = zf.decode_attn(gc, q, table, lens, layer.scale, kernel=kernel)
    torch.cuda.synchronize()
    assert gc.status_word() == 0
    oc = H.oracle_cache_from(layer, O)
    ref_out, ref_lse = O.decode_attention(H.np_bits(layer.q), oc, layer.page_table.numpy(), layer.seq_lens.numpy(),
                                          layer.scale)
    H.compare_attention(out, lse, ref_out, ref_lse)
    assert torch.equal(o1, out) and torch.equal(l1, lse)


def test_wait_limits_out_of_range_are_rejected(zf):
    w = I.Workload("case", 1, 8, 2, 16, 64, seed=6)
    layer = I.make_layer(w)
    gc = H.gpu_cache_from(layer, zf)
    dev = torch.device("cuda")
    args = (gc, layer.q.to(dev), layer.page_table.to(dev), layer.seq_lens.to(dev), layer.scale)
    for limit, delay in ((999, 0), (3_000_000_000, 0), (1_000_000, 3_000_000_000)):
        with pytest.raises(zf.ZfError, match="invalid argument"):
            zf.decode_attn_wait_test(*args, wait_limit_ns=limit, publish_delay_ns=delay)
