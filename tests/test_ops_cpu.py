"""The allocating wrappers' forward workspace handling, without a GPU: the
C call is replaced by a recorder, the workspace-size query is the library's
own (it needs no device).  `ops.norm_fwd` queries and allocates a workspace
only when the call writes no row statistics, and passes a caller's
workspace through as given."""
import pytest
import torch


@pytest.fixture(scope="module")
def ops():
    from rmsnorm_fp8_quantization_gb300 import _build
    _build.build()
    from rmsnorm_fp8_quantization_gb300 import ops as o
    return o


@pytest.fixture
def calls(ops, monkeypatch):
    rec = []
    real_query = ops.G.gbn_norm_fwd_workspace_size

    def query(*args):
        rec.append(("query", args))
        return real_query(*args)

    def fwd(*args, **kw):
        # workspace, workspace_bytes are the 13th and 14th arguments
        rec.append(("fwd", args[12], args[13]))
        return ops.G.GBN_OK

    monkeypatch.setattr(ops.G, "gbn_norm_fwd_workspace_size", query)
    monkeypatch.setattr(ops.G, "gbn_norm_fwd", fwd)
    return rec


def _outputs(ops, rows, hidden, training, layout="colwise"):
    return ops.fwd_outputs(rows, hidden, torch.bfloat16, "rmsnorm", "delayed", layout, "cpu",
                           training)


def _call(ops, rows, hidden, training, layout="colwise", workspace=None):
    x = torch.zeros(rows, hidden, dtype=torch.bfloat16)
    g = torch.ones(hidden, dtype=torch.bfloat16)
    s = torch.ones(1)
    ops.norm_fwd(x, g, None, norm="rmsnorm", scaling="delayed", layout=layout, scale=s,
                 outputs=_outputs(ops, rows, hidden, training, layout), training=training,
                 workspace=workspace)


def test_no_workspace_when_statistics_are_written(ops, calls):
    _call(ops, 64, 49152, training=True)
    assert [c[0] for c in calls] == ["fwd"]
    assert calls[0][1] is None and calls[0][2] == 0


def test_workspace_for_long_columnwise_rows_without_statistics(ops, calls):
    _call(ops, 64, 49152, training=False)
    assert [c[0] for c in calls] == ["query", "fwd"]
    ws, nbytes = calls[1][1], calls[1][2]
    assert ws is not None and ws.dtype == torch.uint8 and nbytes == ws.numel() == 256


def test_none_for_short_rows_without_statistics(ops, calls):
    _call(ops, 64, 4096, training=False)
    assert [c[0] for c in calls] == ["query", "fwd"]
    assert calls[1][1] is None and calls[1][2] == 0


def test_callers_workspace_passed_through(ops, calls):
    mine = torch.empty(1000, dtype=torch.uint8)
    _call(ops, 64, 49152, training=False, workspace=mine)
    assert [c[0] for c in calls] == ["fwd"]
    assert calls[0][1] is mine and calls[0][2] == 1000
