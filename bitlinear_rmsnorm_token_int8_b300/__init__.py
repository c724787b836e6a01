"""BitNet b1.58 BitLinear forward on B300 (sm_103a): placeholder, binding added next."""
