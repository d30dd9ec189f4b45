"""GB300-native EP-MoE all-to-all (Reverse All2All combine and dispatch) over an
emulated symmetric heap."""
