"""GB300-native speculative-decoding verify, SMC-SD reweight / resample and PACER stop rule.

The compute path is the CUDA library ``libsmcsd.so`` (C ABI in ``include/smcsd.h``); the
functions exported here are its ctypes binding (``_binding``), loaded on first use. Build the
library with ``smc_reweight_resample_gb300.build.build()``. ``synth`` holds the seeded input
generators.
"""
_API = {
    "sd_verify", "smc_reweight", "smc_ess_resample", "kv_pagetable_remap", "pacer_block_stop",
    "smc_step", "Workspace", "workspace_size", "check_status", "status_string", "SMCSDError",
    "load", "OP_SD_VERIFY", "OP_SMC_REWEIGHT", "OP_SMC_STEP", "OP_ESS_RESAMPLE",
    "OP_PAGETABLE_REMAP", "OP_PACER_BLOCK_STOP", "LIB_PATH",
}

__all__ = sorted(_API)


def __getattr__(name):
    if name in _API:
        from . import _binding

        return getattr(_binding, name)
    raise AttributeError(name)
