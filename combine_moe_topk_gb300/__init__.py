"""GB300-native MoE token path: top-k gating, dispatch layout, dispatch,
combine and their backward duals, behind a C ABI (``libmoe_gb300.so``)."""
