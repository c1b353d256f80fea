"""UltraEP per-microbatch, per-layer expert-parallel balancing hot path for B300.

The compute path is the C-ABI library built from ``csrc/`` (hand-written CUDA
for sm_103a); ``ultraep`` is its thin Python binding.  ``workload`` draws the
seeded synthetic inputs and ``quality`` holds the host-side plan-quality
metrics.  The binding's names are re-exported lazily so that importing the
workload or quality helpers does not need the compiled library.
"""
_BINDING_NAMES = ("ep_count", "ep_plan", "ep_plan_ex", "ep_reroute", "ep_balance", "ep_permute", "ep_unpermute",
                  "ep_combine", "ep_stage",
                  "ep_count_workspace_bytes", "ep_status_str", "Domain", "EpError")


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import ultraep
        return getattr(ultraep, name)
    raise AttributeError(name)
